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
// Section 0x06.1C: dQ reduces over key tiles, dK/dV over query tiles, and no
// single owner makes all three single-writer.  Instead of the column owner
// with fp32 atomic dQ of 0x06.1D, each reduction gets its own owner (both
// owners are named in 0x06.1C / 0x06.1I; the scores are recomputed by each):
//   1. bwd_preprocess_kernel: D = rowsum(dO * O) in fp32;
//   2. bwd_dkdv_kernel, the column owner: one CTA per 128-key tile of one
//      (batch, KV head) loops over every visible 128-row query block of EVERY
//      query head that reads this KV head; dK and dV accumulate in tensor
//      memory, so the grouped-query sum of 0x06.1H happens in the
//      accumulator (no expanded per-query-head buffers, no group-sum pass);
//   3. bwd_dq_kernel, the row owner: one CTA per 128-row query block of one
//      (batch, query head) loops over every visible key tile; dQ accumulates
//      in tensor memory.
// Every gradient element has one writer and a fixed summation order, so the
// result is bitwise repeatable and no fp32 scratch beyond D is needed.  The
// price is two more 128 x 128 products per (query block, key tile) pair
// (S and dP are formed by both owners): seven instead of five.
//
// Column owner, per query block t (128 rows of query head h); the key axis
// is the TMEM lane axis, each thread of the two "P" warpgroups owns one key
// row and 64 of the block's 128 query columns:
//     S^T  = K Q_t^T       A = K (smem, K-major),    B = Q_t (smem, K-major)
//     dP^T = V dO_t^T      A = V (smem, K-major),    B = dO_t (smem, K-major)
//     dV  += P^T dO_t      A = P^T (tensor memory),  B = dO_t (smem, MN-major)
//     dK  += dS^T Q_t      A = dS^T (tensor memory), B = Q_t (smem, MN-major)
//   P^T / dS^T (input dtype) overwrite the fp32 S^T / dP^T they came from.
//   TMEM: dV [0,128), dK [128,256), S^T/P^T [256,384), dP^T/dS^T [384,512).
//
// Row owner, per key tile j; the query axis is the TMEM lane axis, each
// thread of the two softmax warpgroups owns one query row and 64 of the
// tile's 128 keys:
//     S    = Q K_j^T       A = Q (tensor memory),    B = K_j (smem, K-major)
//     dP   = dO V_j^T      A = dO (tensor memory),   B = V_j (smem, K-major)
//     dQ  += dS K_j        A = dS (smem, K-major),   B = K_j (smem, MN-major)
//   Q and dO are written to tensor memory once per CTA; dS (input dtype) is
//   staged in shared memory, so dP(j+1) can be issued as soon as dP(j) is in
//   registers, while dS(j) is still being formed.
//   TMEM: dQ [0,128), S [128,256), dP [256,384), Q [384,448), dO [448,512).
//
// A 128 x 128 x 16 MMA with both operands in shared memory is bound by the
// shared-memory operand reads (two 4 KiB operands per ~70 cycles, measured);
// every product above with an operand in tensor memory reads only one.
//
// Roles (384 threads, three warpgroups; setmaxnreg 184 / 184 / 136):
//   warps 0-7   two compute warpgroups (columns [0,64) and [64,128))
//   warp  8     loader (TMA; the column owner's loader lanes also stage the
//               block's row statistics in shared memory)
//   warp  9     TMEM allocation; lane 0 issues every MMA and commit
//
// Causal (bottom-right delta = Sk - Sq): tiles wholly in the future are never
// visited; tiles crossing the diagonal and the key / query tails are masked
// element-wise before the exponential.
#include <cuda_runtime.h>

#include "gbattn_internal.h"
#include "gbattn_ptx.cuh"

namespace gbattn {
namespace {

constexpr int kT = 128;      // rows (keys or queries) per tile; head dimension D = 64 or 128
constexpr int kThreads = 384;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kMmaWarpY = 10;  // column owner, d = 128: issuer of the dP^T / dK chain
constexpr int kRegsCompute = 184, kRegsCtl = 136;
static_assert(2 * 128 * kRegsCompute + 128 * kRegsCtl <= kThreads * 168, "register split");
constexpr float kLog2e = 1.4426950408889634f;

constexpr int kBlock = kT * 128;         // 16 KiB: 128 rows x one 128-byte (64-element) column block
constexpr int kDSBytes = kT * kT * 2;    // 32 KiB: a 128 x 128 16-bit dS tile

struct BwdParams {
  const float* lse;   // [B,H,Sq] natural log
  const float* Dvec;  // [B,H,Sq]
  const void* q;      // [B,H,Sq,D]   (row owner: Q and dO rows into TMEM)
  const void* dout;
  void* dq;           // [B,H,Sq,D]
  void* dk;           // [B,Hkv,Sk,D]
  void* dv;
  int B, H, Hkv, Sq, Sk, g;
  int n_ktiles, n_qtiles, head_group, delta;
  float scale, scale_log2;
  int* status;
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         int* status) {
  return bounded_wait(bar, parity, abort_flag, status, kStatusTimeoutBwd);
}

// Descriptor K-steps.  K-major: a step of 16 elements adds 32 bytes inside a
// 128-byte row, or jumps a 16 KiB column block.  MN-major (leading offset =
// 16 KiB between 64-element column blocks, stride offset = 8 rows of 128
// bytes): a step of 16 rows adds 2048 bytes.
__device__ __forceinline__ uint64_t kstep_kmajor(int kk) {
  return static_cast<uint64_t>(((kk / 4) * kBlock + (kk % 4) * 32) >> 4);
}
__device__ __forceinline__ uint64_t kstep_mnmajor(int kk) { return static_cast<uint64_t>((kk * 2048) >> 4); }

// Rounds 32 fp32 values x[base .. base+32) to 16 packed 16-bit pairs
// (element 2i in the low half).
template <bool BF16>
__device__ __forceinline__ void pack32(const float (&x)[64], int base, uint32_t (&pk)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = pack2<BF16>(x[base + 2 * i], x[base + 2 * i + 1]);
}

// =========================================================================
// Column owner: dK, dV.
// =========================================================================
template <int D>
struct ColCfg {
  static constexpr int kTileBytes = kT * D * 2;          // a 128-row tile of Q, dO, K or V
  static constexpr int kStages = (D == 128) ? 2 : 4;     // Q/dO stages
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;                 // kStages tiles
  static constexpr int kOffDO = kOffQ + kStages * kTileBytes;      // kStages tiles
  // P^T (128 keys x 128 queries, K-major A of dV) is staged in shared memory
  // when four Q/dO stages leave room for it (d = 64): S^T(t+1) then follows
  // as soon as S^T(t) has been copied to registers.  With two stages (d = 128)
  // the next block's Q/dO load would sit on that path, so P^T overwrites S^T
  // in tensor memory and S^T(t+1) follows dV(t).
  static constexpr bool kPTSmem = (D == 64);
  static constexpr int kOffPT = kOffDO + kStages * kTileBytes;
  static constexpr int kOffStats = kOffPT + (kPTSmem ? kT * kT * 2 : 0);  // kStages x (128 lse2 + 128 D) fp32
  static constexpr int kOffBars = kOffStats + kStages * 2 * kT * 4;
  // Alignment slack for the 1024-byte swizzle atoms only where it fits; without
  // it the kernel checks that the dynamic shared memory base is aligned.
  static constexpr int kSlack = (1024 + kOffBars + 256 <= 232448) ? 1024 : 0;
  static constexpr int kSmemBytes = kSlack + kOffBars + 256;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // TMEM: dV, dK (D columns each), S^T (-> P^T when kPTSmem is false) and
  // dP^T/dS^T (128 each)
  static constexpr uint32_t kColDV = 0, kColDK = D, kColX = 2 * D, kColY = 2 * D + 128;

  struct __align__(8) Bars {
    uint64_t kv_full;
    uint64_t qd_full[kStages];
    uint64_t qd_empty[kStages];
    uint64_t s_full, s_free, dp_full;
    uint64_t p_full, ds_full;
    uint64_t dv_done, dk_done;
    uint64_t acc_done;
    uint32_t tmem_base;
    int abort_flag;
  };
  static_assert(sizeof(Bars) <= 256, "barrier block");
};

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v,
                    const __grid_constant__ CUtensorMap tmap_do, const __grid_constant__ CUtensorMap tmap_dk,
                    const __grid_constant__ CUtensorMap tmap_dv, const BwdParams p) {
  using C = ColCfg<D>;
  using Bars = typename C::Bars;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (C::kSlack == 0 && (smem_u32(smem_raw) & 1023u) != 0) {  // uniform over the CTA
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kStatusSmemAlign);
    return;
  }
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBars);
  float* stats = reinterpret_cast<float*>(smem + C::kOffStats);  // [stage][lse2 128 | D 128]
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // ---- work unit: (batch * Hkv + kv head, key tile).  CTAs run in groups of
  // p.head_group KV heads (their Q/dO working set stays in L2); inside a
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
  const int k0 = jt * kT;
  const int nqb = p.n_qtiles;
  int i_start = 0;
  if (CAUSAL) {
    const int q_min = k0 - p.delta;  // first query row that sees key k0
    i_start = q_min <= 0 ? 0 : (q_min >= p.Sq ? nqb : q_min / kT);
  }
  const int n_blk = nqb - i_start;
  const int T = p.g * n_blk;  // query blocks this CTA visits

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->qd_full[s], 1 + 32);  // TMA arrive + 32 lanes' stat stores
      mbar_init(&bars->qd_empty[s], C::kPTSmem ? 1 : 2);  // d = 128: released by both issuers
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 256);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 256);
    mbar_init(&bars->ds_full, 256);
    mbar_init(&bars->dv_done, 1);
    mbar_init(&bars->dk_done, 1);
    mbar_init(&bars->acc_done, C::kPTSmem ? 1 : 2);
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
    q0 = (i_start + (t - hh * n_blk)) * kT;
  };

  if (warp >= kLoadWarp) {
    regs_dec<kRegsCtl>();
    if (warp == kLoadWarp && T > 0) {
      // ============================================================== loader
      const uint64_t once = policy_evict_first();  // K/V: read by this CTA only
      const uint64_t reuse = policy_evict_last();  // Q/dO: re-read by every key tile
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->kv_full, 2 * C::kTileBytes);
        for (int cb = 0; cb < D / 64; ++cb) {
          tma_load_3d(smem + C::kOffK + cb * kBlock, &tmap_k, &bars->kv_full, cb * 64, k0, bkv, once);
          tma_load_3d(smem + C::kOffV + cb * kBlock, &tmap_v, &bars->kv_full, cb * 64, k0, bkv, once);
        }
      }
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % C::kStages;
        const bool ok = wait_bar(&bars->qd_empty[s], ((t / C::kStages) & 1) ^ 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) break;
        int h, q0;
        block_coords(t, h, q0);
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->qd_full[s], 2 * C::kTileBytes);
          for (int cb = 0; cb < D / 64; ++cb) {
            tma_load_3d(smem + C::kOffQ + s * C::kTileBytes + cb * kBlock, &tmap_q, &bars->qd_full[s], cb * 64,
                        q0, b * p.H + h, reuse);
            tma_load_3d(smem + C::kOffDO + s * C::kTileBytes + cb * kBlock, &tmap_do, &bars->qd_full[s],
                        cb * 64, q0, b * p.H + h, reuse);
          }
        }
        // Row statistics of the block: LSE in base 2 (+inf for rows past Sq
        // and rows with no visible key, so that their P is exactly 0) and D.
        const long long row0 = (static_cast<long long>(b) * p.H + h) * p.Sq;
        float* st = stats + s * 2 * kT;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = lane + 32 * u;
          const int row = q0 + c;
          float l2 = INFINITY, dv = 0.f;
          if (row < p.Sq) {
            const float lse = p.lse[row0 + row];
            if (lse != -INFINITY) l2 = lse * kLog2e;
            dv = p.Dvec[row0 + row];
          }
          st[c] = l2;
          st[kT + c] = dv;
        }
        mbar_arrive(&bars->qd_full[s]);
        issued = t + 1;
      }
      if (lane == 0) {
        // Drain: every copy this warp issued must land before exit.
        int dummy = 0;
        volatile int* no_abort = reinterpret_cast<volatile int*>(&dummy);
        bounded_wait(&bars->kv_full, 0, no_abort, p.status, kStatusTimeoutDrain);
        for (int t = max(0, issued - C::kStages); t < issued; ++t)
          bounded_wait(&bars->qd_full[t % C::kStages], (t / C::kStages) & 1, no_abort, p.status,
                       kStatusTimeoutDrain);
      }
      __syncwarp();
    } else if (warp == kMmaWarp || (!C::kPTSmem && warp == kMmaWarpY)) {
      // ============================================================== MMA issuers
      // d = 64: warp 9 issues everything.  d = 128: warp 9 issues the S^T / dV
      // chain and warp 10 the dP^T / dK chain, so that neither waits behind
      // the other's barrier (P^T and dS^T overwrite S^T and dP^T in TMEM).
      const bool chain_x = warp == kMmaWarp;
      if (lane == 0 && T > 0) {
        constexpr uint32_t kIdSS = idesc_f16(BF16, false, false, 128, 128);  // S^T, dP^T
        constexpr uint32_t kIdTS = idesc_f16(BF16, false, true, 128, D);     // dV, dK
        const uint64_t dK_A = smem_desc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
        const uint64_t dV_A = smem_desc_sw128(smem_u32(smem + C::kOffV), 16, 1024);
        const uint32_t aQ0 = smem_u32(smem + C::kOffQ), aDO0 = smem_u32(smem + C::kOffDO);
        auto issue_ss = [&](uint32_t d_col, uint64_t a_desc, uint32_t b_base) {
          const uint64_t bd = smem_desc_sw128(b_base, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_f16_ss(tmem + d_col, a_desc + kstep_kmajor(kk), bd + kstep_kmajor(kk), kIdSS, kk > 0 ? 1u : 0u);
        };
        // A from tensor memory: 16 query rows (K) = 8 packed columns; rows
        // 0-63 sit in columns [0,32) of the region, rows 64-127 in [64,96).
        auto issue_ts = [&](uint32_t d_col, uint32_t a_col, uint32_t b_base, bool accumulate) {
          const uint64_t bd = smem_desc_sw128(b_base, kBlock, 1024);
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_f16_ts(tmem + d_col, tmem + a_col + (kk / 4) * 64 + (kk % 4) * 8, bd + kstep_mnmajor(kk), kIdTS,
                       (accumulate || kk > 0) ? 1u : 0u);
        };
        bool ok = wait_bar(&bars->kv_full, 0, abort_flag, p.status) &&
                  wait_bar(&bars->qd_full[0], 0, abort_flag, p.status);
        if (ok) {
          tc_fence_after();
          if (chain_x) {
            issue_ss(C::kColX, dK_A, aQ0);
            mma_commit(&bars->s_full);
          }
          if (C::kPTSmem || !chain_x) {
            issue_ss(C::kColY, dV_A, aDO0);
            mma_commit(&bars->dp_full);
          }
        }
        if constexpr (C::kPTSmem) {
          // dV += P^T dO: A = P^T in shared memory (K-major, two 64-query column
          // blocks), B = dO (MN-major).
          const uint64_t pt_desc = smem_desc_sw128(smem_u32(smem + C::kOffPT), 16, 1024);
          auto issue_dv = [&](uint32_t b_base, bool accumulate) {
            const uint64_t bd = smem_desc_sw128(b_base, kBlock, 1024);
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk)
              mma_f16_ss(tmem + C::kColDV, pt_desc + kstep_kmajor(kk), bd + kstep_mnmajor(kk), kIdTS,
                         (accumulate || kk > 0) ? 1u : 0u);
          };
          for (int t = 0; ok && t < T; ++t) {
            const int s = t % C::kStages;
            const uint32_t ph = t & 1;
            const int s1 = (t + 1) % C::kStages;
            // S^T(t+1) as soon as both warpgroups hold S^T(t) in registers (P^T
            // lives in shared memory, so the S^T columns are free then)
            if (t + 1 < T) {
              if (!(ok = wait_bar(&bars->qd_full[s1], ((t + 1) / C::kStages) & 1, abort_flag, p.status))) break;
              if (!(ok = wait_bar(&bars->s_free, ph, abort_flag, p.status))) break;
              tc_fence_after();
              issue_ss(C::kColX, dK_A, aQ0 + s1 * C::kTileBytes);
              mma_commit(&bars->s_full);
            }
            // dV += P^T(t) dO_t
            if (!(ok = wait_bar(&bars->p_full, ph, abort_flag, p.status))) break;
            tc_fence_after();
            issue_dv(aDO0 + s * C::kTileBytes, t > 0);
            mma_commit(&bars->dv_done);
            // dK += dS^T Q_t (the last reader of this Q/dO stage)
            if (!(ok = wait_bar(&bars->ds_full, ph, abort_flag, p.status))) break;
            tc_fence_after();
            issue_ts(C::kColDK, C::kColY, aQ0 + s * C::kTileBytes, t > 0);
            mma_commit(&bars->dk_done);
            mma_commit(&bars->qd_empty[s]);
            // dP^T(t+1) over dS^T(t) once dK has read it
            if (t + 1 < T) {
              if (!(ok = wait_bar(&bars->dk_done, ph, abort_flag, p.status))) break;
              tc_fence_after();
              issue_ss(C::kColY, dV_A, aDO0 + s1 * C::kTileBytes);
              mma_commit(&bars->dp_full);
            }
          }
        } else if (chain_x) {
          for (int t = 0; ok && t < T; ++t) {
            const int s = t % C::kStages;
            const uint32_t ph = t & 1;
            // dV += P^T dO_t (this chain's last reader of the stage)
            if (!(ok = wait_bar(&bars->p_full, ph, abort_flag, p.status))) break;
            tc_fence_after();
            issue_ts(C::kColDV, C::kColX, aDO0 + s * C::kTileBytes, t > 0);
            mma_commit(&bars->dv_done);
            mma_commit(&bars->qd_empty[s]);
            // S^T(t+1) over P^T(t) once dV has read it
            if (t + 1 < T) {
              const int s1 = (t + 1) % C::kStages;
              if (!(ok = wait_bar(&bars->qd_full[s1], ((t + 1) / C::kStages) & 1, abort_flag, p.status))) break;
              if (!(ok = wait_bar(&bars->dv_done, ph, abort_flag, p.status))) break;
              tc_fence_after();
              issue_ss(C::kColX, dK_A, aQ0 + s1 * C::kTileBytes);
              mma_commit(&bars->s_full);
            }
          }
        } else {
          for (int t = 0; ok && t < T; ++t) {
            const int s = t % C::kStages;
            const uint32_t ph = t & 1;
            // dK += dS^T Q_t (this chain's last reader of the stage)
            if (!(ok = wait_bar(&bars->ds_full, ph, abort_flag, p.status))) break;
            tc_fence_after();
            issue_ts(C::kColDK, C::kColY, aQ0 + s * C::kTileBytes, t > 0);
            mma_commit(&bars->dk_done);
            mma_commit(&bars->qd_empty[s]);
            // dP^T(t+1) over dS^T(t) once dK has read it
            if (t + 1 < T) {
              const int s1 = (t + 1) % C::kStages;
              if (!(ok = wait_bar(&bars->qd_full[s1], ((t + 1) / C::kStages) & 1, abort_flag, p.status))) break;
              if (!(ok = wait_bar(&bars->dk_done, ph, abort_flag, p.status))) break;
              tc_fence_after();
              issue_ss(C::kColY, dV_A, aDO0 + s1 * C::kTileBytes);
              mma_commit(&bars->dp_full);
            }
          }
        }
        mma_commit(&bars->acc_done);
        // Every MMA issued must complete before TMEM is released.
        int dummy = 0;
        bounded_wait(&bars->acc_done, 0, reinterpret_cast<volatile int*>(&dummy), p.status,
                     kStatusTimeoutDrain);
      }
      __syncwarp();
    }
  } else {
    // ================================================================ P warpgroups
    regs_inc<kRegsCompute>();
    const int wg = warp / 4;                // query columns [64 wg, 64 wg + 64) of a block
    const int kl = (warp % 4) * 32 + lane;  // key row within the tile (= TMEM lane)
    const int key = k0 + kl;
    const uint32_t lane_off = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t colX = tmem + lane_off + C::kColX + wg * 64;
    const uint32_t colY = tmem + lane_off + C::kColY + wg * 64;
    const float lam = p.scale_log2;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int s = t % C::kStages;
      const uint32_t ph = t & 1;
      int h, q0;
      block_coords(t, h, q0);
      (void)h;
      const int c0 = q0 + wg * 64;  // query row of this warpgroup's first column
      ok = wait_bar(&bars->s_full, ph, abort_flag, p.status) &&
           wait_bar(&bars->qd_full[s], (t / C::kStages) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float4* st_l = reinterpret_cast<const float4*>(stats + s * 2 * kT + wg * 64);
      const float4* st_d = reinterpret_cast<const float4*>(stats + s * 2 * kT + kT + wg * 64);
      // One 64-value register row holds S^T, then P^T, then dS^T.
      float x[64];
      tmem_ld32(colX, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      tmem_ld32(colX + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      tmem_wait_ld();
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      if constexpr (C::kPTSmem) {
        tc_fence_before();
        mbar_arrive(&bars->s_free);  // S^T(t) copied: the issuer may write S^T(t+1)
      }
      // P = 2^(lambda s - LSE log2 e); masked: keys past Sk, and (causal)
      // column c with c0 + c + delta < key.
      const bool need_mask = (k0 + kT > p.Sk) || (CAUSAL && (k0 + kT - 1 > c0 + p.delta));
      const int first_c = (key >= p.Sk) ? 64 : (CAUSAL ? key - p.delta - c0 : 0);
      const float2 lam2 = make_float2(lam, lam);
      if (!need_mask) {  // block-uniform: every block but the diagonal and ragged ones
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 l4 = st_l[c4];  // broadcast read
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int c = 4 * c4 + 2 * i;
            const float2 nl = i ? make_float2(-l4.z, -l4.w) : make_float2(-l4.x, -l4.y);
            const float2 e = ex2_pair(ffma2(make_float2(x[c], x[c + 1]), lam2, nl), c / 2);
            x[c] = e.x;
            x[c + 1] = e.y;
          }
        }
      } else {
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 l4 = st_l[c4];  // broadcast read
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int c = 4 * c4 + 2 * i;
            const float2 nl = i ? make_float2(-l4.z, -l4.w) : make_float2(-l4.x, -l4.y);
            const float2 e = ex2_pair(ffma2(make_float2(x[c], x[c + 1]), lam2, nl), c / 2);
            x[c] = (c < first_c) ? 0.f : e.x;
            x[c + 1] = (c + 1 < first_c) ? 0.f : e.y;
          }
        }
      }
      if constexpr (C::kPTSmem) {
        {
          // P^T row of this key, queries [64 wg, 64 wg + 64): 128 bytes of the
          // warpgroup's column block, 16-byte chunk c at chunk c ^ (key row % 8),
          // once dV(t-1) has read P^T(t-1)
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) pk[i] = pack2<BF16>(x[2 * i], x[2 * i + 1]);
          if (t > 0) {
            ok = wait_bar(&bars->dv_done, (t - 1) & 1, abort_flag, p.status);
            if (!__all_sync(0xffffffffu, ok)) {
              ok = false;
              break;
            }
          }
          uint8_t* pt_row = smem + C::kOffPT + wg * kBlock + kl * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(pt_row + ((c ^ (kl & 7)) << 4)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        fence_proxy_async_smem();  // P^T stores -> visible to the tensor core
        mbar_arrive(&bars->p_full);
      } else {
        {
          uint32_t pk[16];
          pack32<BF16>(x, 0, pk);
          tmem_st16(colX, pk);  // P^T over this warpgroup's own S^T columns
          pack32<BF16>(x, 32, pk);
          tmem_st16(colX + 16, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full);
      }
      // dP^T -> dS^T, 32 columns at a time
      ok = wait_bar(&bars->dp_full, ph, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t w[32];
        tmem_ld32(colY + hf * 32, w);
        tmem_wait_ld();
        reg_fence32(w);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 d4 = st_d[hf * 8 + c4];  // broadcast read
          const int cb = hf * 32 + 4 * c4;
          const float2 a = fmul2(make_float2(x[cb], x[cb + 1]),
                                 fadd2(make_float2(__uint_as_float(w[4 * c4]), __uint_as_float(w[4 * c4 + 1])),
                                       make_float2(-d4.x, -d4.y)));
          const float2 b2 = fmul2(make_float2(x[cb + 2], x[cb + 3]),
                                  fadd2(make_float2(__uint_as_float(w[4 * c4 + 2]), __uint_as_float(w[4 * c4 + 3])),
                                        make_float2(-d4.z, -d4.w)));
          x[cb] = a.x;
          x[cb + 1] = a.y;
          x[cb + 2] = b2.x;
          x[cb + 3] = b2.y;
        }
        uint32_t pk[16];
        pack32<BF16>(x, hf * 32, pk);
        tmem_st16(colY + hf * 16, pk);  // dS^T over dP^T columns already read
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->ds_full);
    }
    // ---- epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK (x tau)
    bool have = ok && T > 0;
    if (have) {
      have = wait_bar(&bars->acc_done, 0, abort_flag, p.status);
      have = __all_sync(0xffffffffu, have);
      tc_fence_after();
    }
    const float mul = wg ? p.scale : 1.f;
    // dV (warpgroup 0) / dK (warpgroup 1) staged in this CTA's own V / K
    // tile (dead once every MMA has completed: acc_done), 128-byte rows with
    // 16-byte chunk c at chunk c ^ (row % 8), and written by TMA (rows past
    // Sk are not written).
    uint8_t* stage = smem + (wg ? C::kOffK : C::kOffV) + kl * 128;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t w[32];
      if (have) {
        tmem_ld32(tmem + lane_off + (wg ? C::kColDK : C::kColDV) + c * 32, w);
        tmem_wait_ld();
        reg_fence32(w);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = 0u;
      }
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        pk[i] = pack2<BF16>(__uint_as_float(w[2 * i]) * mul, __uint_as_float(w[2 * i + 1]) * mul);
      uint8_t* blk = stage + (c / 2) * kBlock;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int ch = (c % 2) * 4 + k;
        *reinterpret_cast<uint4*>(blk + ((ch ^ (kl & 7)) << 4)) =
            make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1 + wg, 128);
    if (warp % 4 == 0 && lane == 0) {
      for (int cb = 0; cb < D / 64; ++cb)
        tma_store_3d(wg ? &tmap_dk : &tmap_dv, smem + (wg ? C::kOffK : C::kOffV) + cb * kBlock, cb * 64, k0, bkv);
      bulk_commit_group();
      bulk_wait_group_read0();
    }
  }

  // ---- teardown: all TMEM traffic done before the allocator warp frees it
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// =========================================================================
// Row owner: dQ.
// =========================================================================
template <int D>
struct RowCfg {
  static constexpr int kTileBytes = kT * D * 2;        // a 128-key tile of K or V
  static constexpr int kStages = (D == 128) ? 3 : 5;   // K/V stages
  static constexpr int kStageBytes = 2 * kTileBytes;   // stage s: K, then V
  static constexpr int kOffKV = 0;
  static constexpr int kOffDS = kOffKV + kStages * kStageBytes;  // dS, K-major A of the dQ product
  static constexpr int kOffBars = kOffDS + kDSBytes;
  static constexpr int kSmemBytes = 1024 + kOffBars + 256;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // TMEM: dQ (D columns), S and dP (128 each), Q and dO (D/2 packed columns each)
  static constexpr uint32_t kColDQ = 0, kColS = D, kColP = D + 128, kColQ = D + 256, kColDO = D + 256 + D / 2;

  struct __align__(8) Bars {
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t qo_ready;
    uint64_t s_full, s_free;
    uint64_t dp_full, dp_free;
    uint64_t ds_full, ds_free;
    uint64_t acc_done;
    uint32_t tmem_base;
    int abort_flag;
  };
  static_assert(sizeof(Bars) <= 256, "barrier block");
};

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ CUtensorMap tmap_dq, const BwdParams p) {
  using C = RowCfg<D>;
  using Bars = typename C::Bars;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBars);
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // ---- work unit: (batch * H + head, query block).  Groups of p.head_group
  // heads (their K/V stay in L2); inside a group the query blocks descend
  // (causal: the blocks with the most key tiles first) and heads vary
  // fastest (query heads of one KV head run side by side).
  const int BH = p.B * p.H;
  const int group = blockIdx.x / (p.head_group * p.n_qtiles);
  const int heads_here = min(p.head_group, BH - group * p.head_group);
  const int r_in = blockIdx.x - group * p.head_group * p.n_qtiles;
  const int bh = group * p.head_group + r_in % heads_here;
  const int it = p.n_qtiles - 1 - r_in / heads_here;
  const int b = bh / p.H;
  const int h = bh % p.H;
  const int kvh = h / p.g;
  const int q0 = it * kT;
  int n = p.n_ktiles;  // key tiles this block visits
  if (CAUSAL) {
    const int lim = min(q0 + kT - 1, p.Sq - 1) + p.delta;  // largest visible key of the block
    n = lim < 0 ? 0 : min(n, lim / kT + 1);
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->qo_ready, 256);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 256);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->dp_free, 256);
    mbar_init(&bars->ds_full, 256);
    mbar_init(&bars->ds_free, 1);
    mbar_init(&bars->acc_done, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp >= kLoadWarp) {
    regs_dec<kRegsCtl>();
    if (warp == kLoadWarp) {
      // ============================================================== loader
      if (lane == 0 && n > 0) {
        const uint64_t keep = policy_evict_last();  // K/V: re-read by every query block
        int issued = 0;
        for (int j = 0; j < n; ++j) {
          const int s = j % C::kStages;
          if (!wait_bar(&bars->kv_empty[s], ((j / C::kStages) & 1) ^ 1, abort_flag, p.status)) break;
          uint8_t* dst = smem + C::kOffKV + s * C::kStageBytes;
          mbar_arrive_expect_tx(&bars->kv_full[s], 2 * C::kTileBytes);
          for (int cb = 0; cb < D / 64; ++cb) {
            tma_load_3d(dst + cb * kBlock, &tmap_k, &bars->kv_full[s], cb * 64, j * kT, b * p.Hkv + kvh, keep);
            tma_load_3d(dst + C::kTileBytes + cb * kBlock, &tmap_v, &bars->kv_full[s], cb * 64, j * kT,
                        b * p.Hkv + kvh, keep);
          }
          issued = j + 1;
        }
        int dummy = 0;
        volatile int* no_abort = reinterpret_cast<volatile int*>(&dummy);
        for (int j = max(0, issued - C::kStages); j < issued; ++j)
          bounded_wait(&bars->kv_full[j % C::kStages], (j / C::kStages) & 1, no_abort, p.status, kStatusTimeoutDrain);
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // ============================================================== MMA issuer
      if (lane == 0 && n > 0) {
        constexpr uint32_t kIdK = idesc_f16(BF16, false, false, 128, 128);  // S, dP (B K-major)
        constexpr uint32_t kIdMN = idesc_f16(BF16, false, true, 128, D);    // dQ (B MN-major)
        const uint32_t aKV0 = smem_u32(smem + C::kOffKV);
        // A from tensor memory: Q / dO rows hold d along 64 packed columns, a
        // K-step of 16 elements = 8 columns.
        auto issue_scores = [&](uint32_t d_col, uint32_t a_col, uint32_t b_base) {
          const uint64_t bd = smem_desc_sw128(b_base, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_f16_ts(tmem + d_col, tmem + a_col + kk * 8, bd + kstep_kmajor(kk), kIdK, kk > 0 ? 1u : 0u);
        };
        const uint64_t dDS_A = smem_desc_sw128(smem_u32(smem + C::kOffDS), 16, 1024);
        auto issue_dq = [&](uint32_t b_base, bool accumulate) {
          const uint64_t bd = smem_desc_sw128(b_base, kBlock, 1024);
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_f16_ss(tmem + C::kColDQ, dDS_A + kstep_kmajor(kk), bd + kstep_mnmajor(kk), kIdMN,
                       (accumulate || kk > 0) ? 1u : 0u);
        };
        bool ok = wait_bar(&bars->qo_ready, 0, abort_flag, p.status) &&
                  wait_bar(&bars->kv_full[0], 0, abort_flag, p.status);
        if (ok) {
          tc_fence_after();
          issue_scores(C::kColS, C::kColQ, aKV0);
          mma_commit(&bars->s_full);
          issue_scores(C::kColP, C::kColDO, aKV0 + C::kTileBytes);
          mma_commit(&bars->dp_full);
        }
        for (int j = 0; ok && j < n; ++j) {
          const int s = j % C::kStages;
          const uint32_t ph = j & 1;
          if (j + 1 < n) {
            const int s1 = (j + 1) % C::kStages;
            if (!(ok = wait_bar(&bars->kv_full[s1], ((j + 1) / C::kStages) & 1, abort_flag, p.status))) break;
            // S(j+1) once both warpgroups hold S(j) in registers
            if (!(ok = wait_bar(&bars->s_free, ph, abort_flag, p.status))) break;
            tc_fence_after();
            issue_scores(C::kColS, C::kColQ, aKV0 + s1 * C::kStageBytes);
            mma_commit(&bars->s_full);
            // dP(j+1) once both warpgroups hold dP(j) in registers
            if (!(ok = wait_bar(&bars->dp_free, ph, abort_flag, p.status))) break;
            tc_fence_after();
            issue_scores(C::kColP, C::kColDO, aKV0 + s1 * C::kStageBytes + C::kTileBytes);
            mma_commit(&bars->dp_full);
          }
          // dQ += dS(j) K_j
          if (!(ok = wait_bar(&bars->ds_full, ph, abort_flag, p.status))) break;
          tc_fence_after();
          issue_dq(aKV0 + s * C::kStageBytes, j > 0);
          mma_commit(&bars->ds_free);
          mma_commit(&bars->kv_empty[s]);
        }
        mma_commit(&bars->acc_done);
        int dummy = 0;
        bounded_wait(&bars->acc_done, 0, reinterpret_cast<volatile int*>(&dummy), p.status,
                     kStatusTimeoutDrain);
      }
      __syncwarp();
    }
  } else {
    // ================================================================ softmax warpgroups
    regs_inc<kRegsCompute>();
    const int wg = warp / 4;                // keys [64 wg, 64 wg + 64) of a tile
    const int rl = (warp % 4) * 32 + lane;  // query row within the block (= TMEM lane)
    const int q_row = q0 + rl;
    const bool row_ok = q_row < p.Sq;
    const uint32_t lane_off = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const long long grow = (static_cast<long long>(b) * p.H + h) * p.Sq + (row_ok ? q_row : 0);
    // The row's Q (warpgroup 0) or dO (warpgroup 1) into tensor memory: the
    // 16-bit pairs in memory are already the packed column words.
    {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(wg ? p.dout : p.q) + grow * D);
      const uint32_t colA = tmem + lane_off + (wg ? C::kColDO : C::kColQ);
#pragma unroll
      for (int half = 0; half < D / 64; ++half) {  // 32 packed columns = 64 elements each
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = row_ok ? src[half * 8 + i] : make_uint4(0u, 0u, 0u, 0u);
          w[4 * i] = v.x, w[4 * i + 1] = v.y, w[4 * i + 2] = v.z, w[4 * i + 3] = v.w;
        }
        tmem_st32(colA + half * 32, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->qo_ready);
    }
    float l2 = INFINITY, Dr = 0.f;  // rows past Sq / with no visible key: P = 0
    if (row_ok) {
      const float lse = p.lse[grow];
      if (lse != -INFINITY) l2 = lse * kLog2e;
      Dr = p.Dvec[grow];
    }
    const float lam = p.scale_log2;
    const uint32_t colS = tmem + lane_off + C::kColS + wg * 64;
    const uint32_t colP = tmem + lane_off + C::kColP + wg * 64;
    uint8_t* ds_row = smem + C::kOffDS + wg * kBlock + rl * 128;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const uint32_t ph = j & 1;
      const int kb = j * kT + wg * 64;  // key of this warpgroup's first column
      ok = wait_bar(&bars->s_full, ph, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[64];
      tmem_ld32(colS, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      tmem_ld32(colS + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      tmem_wait_ld();
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      tc_fence_before();
      mbar_arrive(&bars->s_free);
      // P = 2^(lambda s - LSE log2 e); masked: keys past Sk and (causal)
      // keys later than q_row + delta, i.e. columns c > last_c.
      const int last_vis = CAUSAL ? min(p.Sk - 1, q_row + p.delta) : p.Sk - 1;
      const int last_c = last_vis - kb;
      const bool need_mask = last_c < 63;
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float2 e = ex2_pair(ffma2(make_float2(x[c], x[c + 1]), make_float2(lam, lam), make_float2(-l2, -l2)), c / 2);
        x[c] = (need_mask && c > last_c) ? 0.f : e.x;
        x[c + 1] = (need_mask && c + 1 > last_c) ? 0.f : e.y;
      }
      ok = wait_bar(&bars->dp_full, ph, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t w[32];
        tmem_ld32(colP + hf * 32, w);
        tmem_wait_ld();
        reg_fence32(w);
        if (hf == 1) {
          tc_fence_before();
          mbar_arrive(&bars->dp_free);  // dP(j+1) may now overwrite the columns
        }
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 v = fmul2(make_float2(x[hf * 32 + i], x[hf * 32 + i + 1]),
                                 fadd2(make_float2(__uint_as_float(w[i]), __uint_as_float(w[i + 1])), make_float2(-Dr, -Dr)));
          x[hf * 32 + i] = v.x;
          x[hf * 32 + i + 1] = v.y;
        }
      }
      // dS row into shared memory (column block wg, row rl; 16-byte chunk c
      // at chunk c ^ (rl % 8)) once the dQ product of tile j-1 has read it.
      if (j > 0) {
        ok = wait_bar(&bars->ds_free, (j - 1) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
      }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t pk[16];
        pack32<BF16>(x, hf * 32, pk);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int cc = hf * 4 + ch;
          *reinterpret_cast<uint4*>(ds_row + ((cc ^ (rl & 7)) << 4)) =
              make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->ds_full);
    }
    // ---- epilogue: dQ row (x tau); warpgroup wg writes columns [wg D/2, (wg + 1) D/2)
    bool have = ok && n > 0;
    if (have) {
      have = wait_bar(&bars->acc_done, 0, abort_flag, p.status);
      have = __all_sync(0xffffffffu, have);
      tc_fence_after();
    }
    // dQ staged in the first K slot of the ring (every load has been consumed
    // and every MMA has completed: acc_done), 128-byte rows with 16-byte
    // chunk c at chunk c ^ (row % 8), and written by TMA (rows past Sq are
    // not written).
    uint8_t* stage = smem + C::kOffKV + rl * 128;
#pragma unroll 1
    for (int c = 0; c < D / 64; ++c) {
      uint32_t w[32];
      if (have) {
        tmem_ld32(tmem + lane_off + C::kColDQ + wg * (D / 2) + c * 32, w);
        tmem_wait_ld();
        reg_fence32(w);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = 0u;
      }
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        pk[i] = pack2<BF16>(__uint_as_float(w[2 * i]) * p.scale, __uint_as_float(w[2 * i + 1]) * p.scale);
      const int col = wg * (D / 2) + c * 32;  // first of these 32 columns
      uint8_t* blk = stage + (col / 64) * kBlock;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int ch = (col % 64) / 8 + k;
        *reinterpret_cast<uint4*>(blk + ((ch ^ (rl & 7)) << 4)) =
            make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1, 256);
    if (warp == 0 && lane == 0) {
      for (int cb = 0; cb < D / 64; ++cb)
        tma_store_3d(&tmap_dq, smem + C::kOffKV + cb * kBlock, cb * 64, q0, b * p.H + h);
      bulk_commit_group();
      bulk_wait_group_read0();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// D[row] = sum_t dO[row,t] * O[row,t] (fp32); 16 threads per row, 8
// elements (16 bytes) each.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const uint16_t* __restrict__ o,
                                                             const uint16_t* __restrict__ dout,
                                                             float* __restrict__ Dvec, long long n_rows) {
  constexpr int kTpr = D / 8;  // threads per row
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long r = tid / kTpr;
  const int part = static_cast<int>(tid % kTpr);
  float acc = 0.f;
  if (r < n_rows) {
    const uint4 a = *reinterpret_cast<const uint4*>(o + r * D + part * 8);
    const uint4 c = *reinterpret_cast<const uint4*>(dout + r * D + part * 8);
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
  }
#pragma unroll
  for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (r < n_rows && part == 0) Dvec[r] = acc;
}

// Heads per L2 scheduling group: about 48 MB of the operands a group re-reads.
int head_group_for(long long per_head_bytes, long long heads) {
  long long hg = (48LL << 20) / (per_head_bytes > 0 ? per_head_bytes : 1);
  if (hg < 1) hg = 1;
  return balanced_head_group(hg, heads, 1);
}

template <int D, bool BF16, bool CAUSAL>
int launch_bwd_t(const BackwardArgs& a) {
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
  if (!make_tmap_3d(&tq, a.q, BF16, D, a.Sq, static_cast<long long>(a.B) * a.H, kT) ||
      !make_tmap_3d(&tdq, a.dq, BF16, D, a.Sq, static_cast<long long>(a.B) * a.H, kT) ||
      !make_tmap_3d(&tdk, a.dk, BF16, D, a.Sk, static_cast<long long>(a.B) * a.Hkv, kT) ||
      !make_tmap_3d(&tdv, a.dv, BF16, D, a.Sk, static_cast<long long>(a.B) * a.Hkv, kT) ||
      !make_tmap_3d(&tdo, a.dout, BF16, D, a.Sq, static_cast<long long>(a.B) * a.H, kT) ||
      !make_tmap_3d(&tk, a.k, BF16, D, a.Sk, static_cast<long long>(a.B) * a.Hkv, kT) ||
      !make_tmap_3d(&tv, a.v, BF16, D, a.Sk, static_cast<long long>(a.B) * a.Hkv, kT))
    return -1;
  const long long n_rows = static_cast<long long>(a.B) * a.H * a.Sq;
  {
    const long long blocks = (n_rows * (D / 8) + 255) / 256;
    if (blocks > 0x7FFFFFFFLL) return -1;
    bwd_preprocess_kernel<D, BF16><<<static_cast<unsigned>(blocks), 256, 0, a.stream>>>(
        static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dout), a.Dvec, n_rows);
  }
  static std::atomic<unsigned long long> col_done{0}, row_done{0};  // per instantiation
  if (!set_smem_limit_once(bwd_dkdv_kernel<D, BF16, CAUSAL>, ColCfg<D>::kSmemBytes, col_done) ||
      !set_smem_limit_once(bwd_dq_kernel<D, BF16, CAUSAL>, RowCfg<D>::kSmemBytes, row_done))
    return -1;
  BwdParams p;
  p.lse = a.lse;
  p.Dvec = a.Dvec;
  p.q = a.q;
  p.dout = a.dout;
  p.dq = a.dq;
  p.dk = a.dk;
  p.dv = a.dv;
  p.B = a.B;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Sk = a.Sk;
  p.g = a.H / a.Hkv;
  p.n_ktiles = (a.Sk + kT - 1) / kT;
  p.n_qtiles = (a.Sq + kT - 1) / kT;
  p.delta = a.Sk - a.Sq;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.status = a.status;
  // column owner: a KV head's group re-reads its query heads' Q and dO
  p.head_group = head_group_for(static_cast<long long>(p.g) * a.Sq * D * 4,
                                static_cast<long long>(a.B) * a.Hkv);
  const long long grid_a = static_cast<long long>(a.B) * a.Hkv * p.n_ktiles;
  if (grid_a > 0x7FFFFFFFLL) return -1;
  bwd_dkdv_kernel<D, BF16, CAUSAL><<<static_cast<unsigned>(grid_a), kThreads, ColCfg<D>::kSmemBytes, a.stream>>>(
      tq, tk, tv, tdo, tdk, tdv, p);
  // row owner: a query head re-reads its KV head's K and V
  BwdParams pr = p;
  pr.head_group = head_group_for(static_cast<long long>(a.Sk) * D * 4, static_cast<long long>(a.B) * a.H);
  const long long grid_b = static_cast<long long>(a.B) * a.H * p.n_qtiles;
  if (grid_b > 0x7FFFFFFFLL) return -1;
  bwd_dq_kernel<D, BF16, CAUSAL><<<static_cast<unsigned>(grid_b), kThreads, RowCfg<D>::kSmemBytes, a.stream>>>(tk, tv, tdq, pr);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_backward(const BackwardArgs& a) {
  if (a.d == 128) {
    if (a.bf16) return a.causal ? launch_bwd_t<128, true, true>(a) : launch_bwd_t<128, true, false>(a);
    return a.causal ? launch_bwd_t<128, false, true>(a) : launch_bwd_t<128, false, false>(a);
  }
  if (a.d != 64) return -1;
  if (a.bf16) return a.causal ? launch_bwd_t<64, true, true>(a) : launch_bwd_t<64, true, false>(a);
  return a.causal ? launch_bwd_t<64, false, true>(a) : launch_bwd_t<64, false, false>(a);
}

}  // namespace gbattn
