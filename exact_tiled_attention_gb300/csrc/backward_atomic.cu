// backward_atomic.cu -- exact attention backward with one owner per key tile
// and dQ accumulated by fp32 atomic adds, on sm_103a.
//
// Same gradients as backward.cu (M4.4 "FlashAttention-2 Work Partitioning and
// the Decode Boundary", 0x06.1A), following the schedule of 0x06.1D: K/V
// column owners commit dK and dV directly, and every (query block, key tile)
// contribution tau dS_ij K_j is added into an fp32 dQ accumulator; atomic
// adds make the sum lossless but not ordered (0x06.1F), so dQ may differ in
// its last bits from call to call.  Three launches in stream order:
//   1. bwd_atomic_prep_kernel: D = rowsum(dO * O) and a zeroed accumulator;
//   2. bwd_atomic_kernel: one CTA per (128-key tile, batch, KV head) over
//      every visible 128-row query block of every query head in the group
//      (the grouped-query sum of dK/dV happens in the accumulator, 0x06.1H);
//   3. bwd_dq_convert_kernel: dQ = tau * accumulator, in the input dtype.
// Against the two-owner kernels this executes five 128 x 128 products per
// (query block, key tile) pair instead of seven and evaluates each
// exponential once; it pays 64 KiB of fp32 adds into L2 per pair.
//
// Per query block t (head dimension 128; keys on the TMEM lane axis, each
// thread of the two compute warpgroups owns one key row and 64 of the
// block's 128 query columns):
//     S^T  = K Q_t^T     A = K (smem, K-major),       B = Q_t (smem, K-major)
//     dP^T = V dO_t^T    A = V (smem, K-major),       B = dO_t (smem, K-major)
//     dV  += P^T dO_t    A = P^T (tensor memory),     B = dO_t (smem, MN-major)
//     dQ^T = K^T dS^T    A = K (smem, MN-major),      B = dS^T (smem, MN-major)
//     dK  += dS^T Q_t    A = dS^T (smem, K-major),    B = Q_t (smem, MN-major)
//   P^T (input dtype) overwrites the fp32 S^T it came from; dS^T is staged in
//   shared memory (the operand of two products); dQ^T lands in the columns of
//   dP^T, which are free once dS^T is formed, and is drained by a warpgroup
//   of its own with coalesced fp32 reductions (a warp adds 32 consecutive
//   head-dimension elements of one query row: 128 bytes).  The reductions are
//   bound by L2 (about 6.5 TB/s of fp32 adds on this GPU), so they stream
//   from warps that nothing else waits on, paced at that rate.
//   TMEM: dV [0,128), dK [128,256), S^T/P^T [256,384), dP^T/dQ^T [384,512).
//
// Roles (512 threads; setmaxnreg 136 / 136 / 88 / 152):
//   warps 0-7   two compute warpgroups (query columns [0,64) and [64,128));
//               per block: dS(t), then P(t+1), so the exponentials of the
//               next block overlap dQ^T(t) and dK(t)
//   warp  8     loader (TMA; its lanes also stage the block's row statistics)
//   warp  9     TMEM allocation; lane 0 issues the S^T -> dV chain
//   warp 10     lane 0 issues the dP^T -> dQ^T -> dK chain
//   warps 12-15 dQ^T drain: TMEM -> registers -> fp32 adds
//
// Causal (bottom-right delta = Sk - Sq) and tails as in backward.cu.
#include <cuda_runtime.h>

#include "gbattn_internal.h"
#include "gbattn_ptx.cuh"

namespace gbattn {
namespace {

constexpr int kT = 128;   // keys per tile, query rows per block
constexpr int kD = 128;   // head dimension
constexpr int kThreads = 512;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarpX = 9;    // TMEM allocation; S^T, dV
constexpr int kMmaWarpY = 10;   // dP^T, dQ^T, dK
constexpr int kDrainWarp0 = 12;  // warps 12-15: dQ^T drain
// setmaxnreg split of the 65,536 registers the launch holds (128 a thread):
// compute warpgroups, control warpgroup, drain warpgroup (all 128 columns of
// a dQ^T row in registers).
constexpr int kRegsCompute = 136, kRegsCtl = 88, kRegsDrain = 152;
static_assert(2 * 128 * kRegsCompute + 128 * kRegsCtl + 128 * kRegsDrain <= kThreads * 128, "register split");
// setmaxnreg.inc may only raise a warp's count and .dec only lower it (the
// launch gives 128 a thread): the roles below use inc / dec accordingly.
static_assert(kRegsCompute >= 128 && kRegsDrain >= 128 && kRegsCtl <= 128, "inc / dec directions");
constexpr float kLog2e = 1.4426950408889634f;

constexpr int kBlock = kT * 128;       // 16 KiB: 128 rows x one 128-byte (64-element) column block
constexpr int kTile = kT * kD * 2;     // 32 KiB: a 128 x 128 16-bit tile
constexpr int kStages = 2;             // Q/dO stages
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kTile;
constexpr int kOffQ = kOffV + kTile;               // kStages tiles
constexpr int kOffDO = kOffQ + kStages * kTile;    // kStages tiles
constexpr int kOffDS = kOffDO + kStages * kTile;   // dS^T: 128 keys x 128 queries, two column blocks
constexpr int kOffStats = kOffDS + kTile;          // kStages x (128 lse2 + 128 D) fp32
constexpr int kOffBars = kOffStats + kStages * 2 * kT * 4;
constexpr int kSmemBytes = kOffBars + 256;  // no room for alignment slack: the base is checked
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kColDV = 0, kColDK = 128, kColX = 256, kColY = 384;

struct __align__(8) Bars {
  uint64_t kv_full;
  uint64_t qd_full[kStages];
  uint64_t qd_empty[kStages];
  uint64_t s_full, dp_full;
  uint64_t p_full, ds_full;
  uint64_t dv_done;
  uint64_t dq_full, dq_free;
  uint64_t acc_done;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct AtomicParams {
  const float* lse;   // [B,H,Sq] natural log
  const float* Dvec;  // [B,H,Sq]
  float* dq_acc;      // [B,H,Sq,128] fp32, zeroed by the prep kernel
  void* dk;           // [B,Hkv,Sk,128]
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

// dQ^T drain pacing: kRedBurst adds per warp, then a pause of kRedPauseNs.
constexpr int kRedBurst = 8;
constexpr unsigned kRedPauseNs = 100;

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

template <bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_atomic_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                      const __grid_constant__ CUtensorMap tmap_dk, const __grid_constant__ CUtensorMap tmap_dv,
                      const AtomicParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {  // uniform over the CTA
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kStatusSmemAlign);
    return;
  }
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBars);
  float* stats = reinterpret_cast<float*>(smem + kOffStats);  // [stage][lse2 128 | D 128]
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // ---- work unit: (batch * Hkv + kv head, key tile), grouped by KV heads so
  // that a group's Q, dO and dQ accumulator stay in L2; inside a group key
  // tiles ascend (causal: the tiles with the most query blocks first) and
  // heads vary fastest.
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
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->qd_full[s], 1 + 32);  // TMA arrive + 32 lanes' stat stores
      mbar_init(&bars->qd_empty[s], 2);      // released by both issuers
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 256);
    mbar_init(&bars->ds_full, 256);
    mbar_init(&bars->dv_done, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 128);
    mbar_init(&bars->acc_done, 2);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
    prefetch_tensormap(&tmap_do);
  }
  if (warp == kMmaWarpX) {
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

  if (warp >= kDrainWarp0) {
    // ================================================================ dQ^T drain
    // dQ^T(t) row kl (head-dim element) over the block's 128 query columns ->
    // registers, columns released, then fp32 adds into the accumulator (a
    // warp adds 32 consecutive head-dim elements of one query row).
    regs_inc<kRegsDrain>();
    const int kl = (warp % 4) * 32 + lane;
    const uint32_t col = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16) + kColY;
    for (int t = 0; t < T; ++t) {
      const bool ok = wait_bar(&bars->dq_full, t & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      uint32_t w[4][32];
#pragma unroll
      for (int i = 0; i < 4; ++i) tmem_ld32(col + 32 * i, w[i]);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 4; ++i) reg_fence32(w[i]);
      tc_fence_before();
      mbar_arrive(&bars->dq_free);
      int h, q0;
      block_coords(t, h, q0);
      float* dst = p.dq_acc + (static_cast<long long>(b * p.H + h) * p.Sq + q0) * kD + kl;
      // The adds are paced at about the rate L2 retires them (8 per warp per
      // 100 ns: about 6.5 TB/s over 152 SMs, measured): issued back to back
      // they fill the load/store queue, and the compute warpgroups' shared
      // memory accesses then wait behind them.
      const int n_rows = min(kT, p.Sq - q0);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (32 * i + c < n_rows) red_add_f32(dst + (32 * i + c) * kD, __uint_as_float(w[i][c]));
          if (c % kRedBurst == kRedBurst - 1) __nanosleep(kRedPauseNs);
        }
    }
  } else if (warp >= kLoadWarp) {
    regs_dec<kRegsCtl>();
    if (warp == kLoadWarp && T > 0) {
      // ============================================================== loader
      const uint64_t once = policy_evict_first();  // K/V: read by this CTA only
      const uint64_t reuse = policy_evict_last();  // Q/dO: re-read by every key tile
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->kv_full, 2 * kTile);
        for (int cb = 0; cb < kD / 64; ++cb) {
          tma_load_3d(smem + kOffK + cb * kBlock, &tmap_k, &bars->kv_full, cb * 64, k0, bkv, once);
          tma_load_3d(smem + kOffV + cb * kBlock, &tmap_v, &bars->kv_full, cb * 64, k0, bkv, once);
        }
      }
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % kStages;
        const bool ok = wait_bar(&bars->qd_empty[s], ((t / kStages) & 1) ^ 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) break;
        int h, q0;
        block_coords(t, h, q0);
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->qd_full[s], 2 * kTile);
          for (int cb = 0; cb < kD / 64; ++cb) {
            tma_load_3d(smem + kOffQ + s * kTile + cb * kBlock, &tmap_q, &bars->qd_full[s], cb * 64, q0,
                        b * p.H + h, reuse);
            tma_load_3d(smem + kOffDO + s * kTile + cb * kBlock, &tmap_do, &bars->qd_full[s], cb * 64, q0,
                        b * p.H + h, reuse);
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
        for (int t = max(0, issued - kStages); t < issued; ++t)
          bounded_wait(&bars->qd_full[t % kStages], (t / kStages) & 1, no_abort, p.status, kStatusTimeoutDrain);
      }
      __syncwarp();
    } else if (warp == kMmaWarpX || warp == kMmaWarpY) {
      // ============================================================== MMA issuers
      const bool chain_x = warp == kMmaWarpX;
      if (lane == 0 && T > 0) {
        constexpr uint32_t kIdS = idesc_f16(BF16, false, false, 128, 128);   // S^T, dP^T
        constexpr uint32_t kIdAcc = idesc_f16(BF16, false, true, 128, kD);   // dV (TS), dK (SS)
        constexpr uint32_t kIdDQ = idesc_f16(BF16, true, true, 128, 128);    // dQ^T: both MN-major
        const uint64_t k_kmaj = smem_desc_sw128(smem_u32(smem + kOffK), 16, 1024);
        const uint64_t v_kmaj = smem_desc_sw128(smem_u32(smem + kOffV), 16, 1024);
        const uint64_t k_mnmaj = smem_desc_sw128(smem_u32(smem + kOffK), kBlock, 1024);
        const uint64_t ds_kmaj = smem_desc_sw128(smem_u32(smem + kOffDS), 16, 1024);
        const uint64_t ds_mnmaj = smem_desc_sw128(smem_u32(smem + kOffDS), kBlock, 1024);
        const uint32_t aQ0 = smem_u32(smem + kOffQ), aDO0 = smem_u32(smem + kOffDO);
        // S^T or dP^T: D = 128 x 128 fp32, K = head dimension
        auto issue_scores = [&](uint32_t d_col, uint64_t a_desc, uint32_t b_base) {
          const uint64_t bd = smem_desc_sw128(b_base, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            mma_f16_ss(tmem + d_col, a_desc + kstep_kmajor(kk), bd + kstep_kmajor(kk), kIdS, kk > 0 ? 1u : 0u);
        };
        bool ok = wait_bar(&bars->kv_full, 0, abort_flag, p.status) &&
                  wait_bar(&bars->qd_full[0], 0, abort_flag, p.status);
        if (ok) {
          tc_fence_after();
          if (chain_x) {
            issue_scores(kColX, k_kmaj, aQ0);
            mma_commit(&bars->s_full);
          } else {
            issue_scores(kColY, v_kmaj, aDO0);
            mma_commit(&bars->dp_full);
          }
        }
        if (chain_x) {
          for (int t = 0; ok && t < T; ++t) {
            const int s = t % kStages;
            const uint32_t ph = t & 1;
            // dV += P^T dO_t: A = P^T in tensor memory (16 query rows = 8
            // packed columns; rows 0-63 in columns [0,32) of the region, rows
            // 64-127 in [64,96)), B = dO_t MN-major.  Last reader of dO_t.
            if (!(ok = wait_bar(&bars->p_full, ph, abort_flag, p.status))) break;
            tc_fence_after();
            {
              const uint64_t bd = smem_desc_sw128(aDO0 + s * kTile, kBlock, 1024);
#pragma unroll
              for (int kk = 0; kk < kT / 16; ++kk)
                mma_f16_ts(tmem + kColDV, tmem + kColX + (kk / 4) * 64 + (kk % 4) * 8, bd + kstep_mnmajor(kk), kIdAcc,
                           (t > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&bars->dv_done);
            mma_commit(&bars->qd_empty[s]);
            // S^T(t+1) over P^T(t) once dV has read it
            if (t + 1 < T) {
              const int s1 = (t + 1) % kStages;
              if (!(ok = wait_bar(&bars->qd_full[s1], ((t + 1) / kStages) & 1, abort_flag, p.status))) break;
              if (!(ok = wait_bar(&bars->dv_done, ph, abort_flag, p.status))) break;
              tc_fence_after();
              issue_scores(kColX, k_kmaj, aQ0 + s1 * kTile);
              mma_commit(&bars->s_full);
            }
          }
        } else {
          for (int t = 0; ok && t < T; ++t) {
            const int s = t % kStages;
            const uint32_t ph = t & 1;
            if (!(ok = wait_bar(&bars->ds_full, ph, abort_flag, p.status))) break;
            tc_fence_after();
            // dQ^T(t) = K^T dS^T over dP^T(t), which every compute thread has read
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk)
              mma_f16_ss(tmem + kColY, k_mnmaj + kstep_mnmajor(kk), ds_mnmaj + kstep_mnmajor(kk), kIdDQ,
                         kk > 0 ? 1u : 0u);
            mma_commit(&bars->dq_full);
            // dK += dS^T Q_t: last reader of dS^T(t) and of Q_t
            {
              const uint64_t bd = smem_desc_sw128(aQ0 + s * kTile, kBlock, 1024);
#pragma unroll
              for (int kk = 0; kk < kT / 16; ++kk)
                mma_f16_ss(tmem + kColDK, ds_kmaj + kstep_kmajor(kk), bd + kstep_mnmajor(kk), kIdAcc,
                           (t > 0 || kk > 0) ? 1u : 0u);
            }
            // (no commit for dK alone: dp_full of the next block, committed after
            // dP^T(t+1), which this thread issues after dK(t), also covers dK(t))
            mma_commit(&bars->qd_empty[s]);
            // dP^T(t+1) over dQ^T(t) once the compute warpgroups drained it
            if (t + 1 < T) {
              const int s1 = (t + 1) % kStages;
              if (!(ok = wait_bar(&bars->qd_full[s1], ((t + 1) / kStages) & 1, abort_flag, p.status))) break;
              if (!(ok = wait_bar(&bars->dq_free, ph, abort_flag, p.status))) break;
              tc_fence_after();
              issue_scores(kColY, v_kmaj, aDO0 + s1 * kTile);
              mma_commit(&bars->dp_full);
            }
          }
        }
        mma_commit(&bars->acc_done);
        // Every MMA issued must complete before TMEM is released.
        int dummy = 0;
        bounded_wait(&bars->acc_done, 0, reinterpret_cast<volatile int*>(&dummy), p.status, kStatusTimeoutDrain);
      }
      __syncwarp();
    }
  } else {
    // ================================================================ compute warpgroups
    regs_inc<kRegsCompute>();
    const int wg = warp / 4;                // query columns [64 wg, 64 wg + 64) of a block
    const int kl = (warp % 4) * 32 + lane;  // TMEM lane: key row of S^T / dP^T, head-dim row of dQ^T
    const int key = k0 + kl;
    const uint32_t lane_off = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t colX = tmem + lane_off + kColX + wg * 64;
    const uint32_t colY = tmem + lane_off + kColY + wg * 64;
    const float lam = p.scale_log2;
    float x[64];  // P of the current block: key row kl, this warpgroup's 64 query columns

    // S^T(t) -> P^T(t): exponentials into x, P^T (input dtype) over this
    // warpgroup's own S^T columns.
    auto phase_p = [&](int t) -> bool {
      const int s = t % kStages;
      int h, q0;
      block_coords(t, h, q0);
      (void)h;
      const int c0 = q0 + wg * 64;  // query row of this warpgroup's first column
      const bool ok = wait_bar(&bars->s_full, t & 1, abort_flag, p.status) &&
                      wait_bar(&bars->qd_full[s], (t / kStages) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) return false;
      tc_fence_after();
      tmem_ld32(colX, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      tmem_ld32(colX + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      tmem_wait_ld();
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      const float4* st_l = reinterpret_cast<const float4*>(stats + s * 2 * kT + wg * 64);
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
      {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack2<BF16>(x[2 * i], x[2 * i + 1]);
        tmem_st16(colX, pk);
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack2<BF16>(x[32 + 2 * i], x[32 + 2 * i + 1]);
        tmem_st16(colX + 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
      return true;
    };

    // dP^T(t) -> dS^T(t) = P (dP - D), into shared memory once dQ^T(t-1) and
    // dK(t-1) have read the previous one -- both are implied by dp_full(t):
    // the dP^T/dS^T chain's thread issues dQ^T(t-1) and dK(t-1) before
    // dP^T(t), and a commit covers every earlier MMA of its thread (one wait
    // fewer per block: 1.6 % causal, 2.1 % GQA); 32 query columns at a time.
    auto phase_ds = [&](int t) -> bool {
      const int s = t % kStages;
      const bool ok = wait_bar(&bars->dp_full, t & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) return false;
      tc_fence_after();
      const float4* st_d = reinterpret_cast<const float4*>(stats + s * 2 * kT + kT + wg * 64);
      // dS^T row of this key, queries [64 wg, 64 wg + 64): 128 bytes of the
      // warpgroup's column block, 16-byte chunk c at chunk c ^ (key row % 8).
      uint8_t* row = smem + kOffDS + wg * kBlock + kl * 128;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t w[32];
        tmem_ld32(colY + hf * 32, w);
        tmem_wait_ld();
        reg_fence32(w);
        uint32_t pk[16];
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
          pk[2 * c4] = pack2<BF16>(a.x, a.y);
          pk[2 * c4 + 1] = pack2<BF16>(b2.x, b2.y);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int chunk = hf * 4 + c;
          *reinterpret_cast<uint4*>(row + ((chunk ^ (kl & 7)) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
      }
      tc_fence_before();         // dP^T reads complete before dQ^T(t) overwrites the columns
      fence_proxy_async_smem();  // dS^T stores -> visible to the tensor core
      mbar_arrive(&bars->ds_full);
      return true;
    };

    bool ok = T > 0 && phase_p(0);
    for (int t = 0; ok && t < T; ++t) {
      if (!(ok = phase_ds(t))) break;
      if (t + 1 < T && !(ok = phase_p(t + 1))) break;
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
    // Sk are not written).  A thread storing its own 256-byte row to global
    // memory instead touches one cache line per lane and store instruction.
    uint8_t* stage = smem + (wg ? kOffK : kOffV) + kl * 128;
#pragma unroll 1
    for (int c = 0; c < kD / 32; ++c) {
      uint32_t w[32];
      if (have) {
        tmem_ld32(tmem + lane_off + (wg ? kColDK : kColDV) + c * 32, w);
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
      for (int cb = 0; cb < kD / 64; ++cb)
        tma_store_3d(wg ? &tmap_dk : &tmap_dv, smem + (wg ? kOffK : kOffV) + cb * kBlock, cb * 64, k0, bkv);
      bulk_commit_group();
      bulk_wait_group_read0();
    }
  }

  // ---- teardown: all TMEM traffic done before the allocator warp frees it
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarpX) tmem_dealloc(tmem, 512);
}

// =========================================================================
// Head dimension 64.  The same schedule; tensor memory and shared memory now
// have room to spare, so dQ (= dS K: query rows on the TMEM lane axis, 64
// head-dim columns) gets columns of its own and dP^T(t+1) no longer waits for
// the drain, and each drain warp stages its 32 query rows of dQ in shared
// memory and adds them into the accumulator with two TMA bulk tensor
// reductions (off the load/store queue the compute warpgroups use).
//   dQ = dS K      A = dS (the dS^T tile read MN-major), B = K (MN-major)
//   TMEM: dV [0,64), dK [64,128), S^T/P^T [128,256), dP^T [256,384), dQ [384,448).
// =========================================================================
namespace d64 {
constexpr int kD = 64;
constexpr int kTile = kT * kD * 2;  // 16 KiB: 128 rows x 64 elements, one column block
constexpr int kStages = 3;          // Q/dO stages
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kTile;
constexpr int kOffQ = kOffV + kTile;
constexpr int kOffDO = kOffQ + kStages * kTile;
constexpr int kOffPS = kOffDO + kStages * kTile;  // dS^T: 128 keys x 128 queries, two column blocks
constexpr int kOffStage = kOffPS + 2 * kBlock;    // dQ staging: per drain warp two 32-row x 32-float boxes
constexpr int kBoxBytes = 32 * 128;               // 4 KiB
constexpr int kOffStats = kOffStage + 8 * kBoxBytes;
constexpr int kOffBars = kOffStats + kStages * 2 * kT * 4;
constexpr int kSmemBytes = kOffBars + 256;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kColDV = 0, kColDK = 64, kColX = 128, kColY = 256, kColQ = 384;
constexpr int kRegsCompute = 160, kRegsCtl = 88, kRegsDrain = 104;
static_assert(2 * 128 * kRegsCompute + 128 * kRegsCtl + 128 * kRegsDrain <= kThreads * 128, "register split");
// directions from the launch's 128: compute inc, control and drain dec
static_assert(kRegsCompute >= 128 && kRegsCtl <= 128 && kRegsDrain <= 128, "inc / dec directions");

struct __align__(8) Bars {
  uint64_t kv_full;
  uint64_t qd_full[kStages];
  uint64_t qd_empty[kStages];
  uint64_t s_full, dp_full, dp_free;
  uint64_t p_full, ds_full;
  uint64_t dv_done, dk_done;
  uint64_t dq_full, dq_free;
  uint64_t acc_done;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barrier block");
}  // namespace d64

template <bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_atomic64_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                        const __grid_constant__ CUtensorMap tmap_dq, const __grid_constant__ CUtensorMap tmap_dk,
                        const __grid_constant__ CUtensorMap tmap_dv, const AtomicParams p) {
  // this kernel's layout (shadows the 128-dim constants)
  constexpr int kD = d64::kD, kTile = d64::kTile, kStages = d64::kStages;
  constexpr int kOffK = d64::kOffK, kOffV = d64::kOffV, kOffQ = d64::kOffQ, kOffDO = d64::kOffDO;
  constexpr int kOffPS = d64::kOffPS, kOffStage = d64::kOffStage, kBoxBytes = d64::kBoxBytes;
  constexpr int kOffStats = d64::kOffStats, kOffBars = d64::kOffBars;
  constexpr uint32_t kColDV = d64::kColDV, kColDK = d64::kColDK, kColX = d64::kColX, kColY = d64::kColY,
                     kColQ = d64::kColQ;
  constexpr int kRegsCompute = d64::kRegsCompute, kRegsCtl = d64::kRegsCtl, kRegsDrain = d64::kRegsDrain;
  using Bars64 = d64::Bars;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {  // uniform over the CTA
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kStatusSmemAlign);
    return;
  }
  Bars64* bars = reinterpret_cast<Bars64*>(smem + kOffBars);
  float* stats = reinterpret_cast<float*>(smem + kOffStats);  // [stage][lse2 128 | D 128]
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // ---- work unit: as the 128-dim kernel
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
    const int q_min = k0 - p.delta;
    i_start = q_min <= 0 ? 0 : (q_min >= p.Sq ? nqb : q_min / kT);
  }
  const int n_blk = nqb - i_start;
  const int T = p.g * n_blk;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->qd_full[s], 1 + 32);  // TMA arrive + 32 lanes' stat stores
      mbar_init(&bars->qd_empty[s], 2);      // released by both issuers
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->dp_free, 256);
    mbar_init(&bars->p_full, 256);
    mbar_init(&bars->ds_full, 256);
    mbar_init(&bars->dv_done, 1);
    mbar_init(&bars->dk_done, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 128);
    mbar_init(&bars->acc_done, 2);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
    prefetch_tensormap(&tmap_do);
  }
  if (warp == kDrainWarp0 && lane == 0) prefetch_tensormap(&tmap_dq);
  if (warp == kMmaWarpX) {
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

  if (warp >= kDrainWarp0) {
    // ================================================================ dQ drain
    // Warp w owns query rows [32 (w % 4), +32) of the block: dQ rows ->
    // registers -> columns released -> its two swizzled 32 x 32 fp32 boxes
    // -> two TMA reduce-adds into the accumulator.
    regs_dec<kRegsDrain>();  // below the launch's 128: setmaxnreg.inc may only raise the count
    const int wq = warp % 4;
    const uint32_t col = tmem + (static_cast<uint32_t>(wq * 32) << 16) + kColQ;
    uint8_t* stage = smem + kOffStage + wq * 2 * kBoxBytes;
    for (int t = 0; t < T; ++t) {
      const bool ok = wait_bar(&bars->dq_full, t & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      uint32_t w[2][32];
      tmem_ld32(col, w[0]);
      tmem_ld32(col + 32, w[1]);
      tmem_wait_ld();
      reg_fence32(w[0]);
      reg_fence32(w[1]);
      tc_fence_before();
      mbar_arrive(&bars->dq_free);
      int h, q0;
      block_coords(t, h, q0);
      const int y = q0 + 32 * wq;
      if (lane == 0 && t > 0) bulk_wait_group_read0();  // this warp's previous boxes are read
      __syncwarp();
      // row `lane` of box j (head-dim columns [32 j, 32 j + 32)): 16-byte chunk c at c ^ (lane % 8)
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(stage + j * kBoxBytes + lane * 128 + ((c ^ (lane & 7)) << 4)) =
              make_uint4(w[j][4 * c], w[j][4 * c + 1], w[j][4 * c + 2], w[j][4 * c + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && y < p.Sq) {
        tma_reduce_add_3d(&tmap_dq, stage, 0, y, b * p.H + h);
        tma_reduce_add_3d(&tmap_dq, stage + kBoxBytes, 32, y, b * p.H + h);
        bulk_commit_group();
      }
    }
    if (lane == 0) bulk_wait_group_read0();
    __syncwarp();
  } else if (warp >= kLoadWarp) {
    regs_dec<kRegsCtl>();
    if (warp == kLoadWarp && T > 0) {
      // ============================================================== loader
      const uint64_t once = policy_evict_first();
      const uint64_t reuse = policy_evict_last();
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->kv_full, 2 * kTile);
        tma_load_3d(smem + kOffK, &tmap_k, &bars->kv_full, 0, k0, bkv, once);
        tma_load_3d(smem + kOffV, &tmap_v, &bars->kv_full, 0, k0, bkv, once);
      }
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % kStages;
        const bool ok = wait_bar(&bars->qd_empty[s], ((t / kStages) & 1) ^ 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) break;
        int h, q0;
        block_coords(t, h, q0);
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->qd_full[s], 2 * kTile);
          tma_load_3d(smem + kOffQ + s * kTile, &tmap_q, &bars->qd_full[s], 0, q0, b * p.H + h, reuse);
          tma_load_3d(smem + kOffDO + s * kTile, &tmap_do, &bars->qd_full[s], 0, q0, b * p.H + h, reuse);
        }
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
        int dummy = 0;
        volatile int* no_abort = reinterpret_cast<volatile int*>(&dummy);
        bounded_wait(&bars->kv_full, 0, no_abort, p.status, kStatusTimeoutDrain);
        for (int t = max(0, issued - kStages); t < issued; ++t)
          bounded_wait(&bars->qd_full[t % kStages], (t / kStages) & 1, no_abort, p.status, kStatusTimeoutDrain);
      }
      __syncwarp();
    } else if (warp == kMmaWarpX || warp == kMmaWarpY) {
      // ============================================================== MMA issuers
      //   X: dV(t) once P^T(t) is written; S^T(t+1) once dV(t) has read it.
      //   Y: dP^T(t+1) once dP^T(t) is in registers; dQ(t), dK(t) once dS^T(t)
      //      is in shared memory (dQ(t) also once dQ(t-1) is drained).
      const bool chain_x = warp == kMmaWarpX;
      if (lane == 0 && T > 0) {
        constexpr uint32_t kIdS = idesc_f16(BF16, false, false, 128, 128);  // S^T, dP^T
        constexpr uint32_t kIdAcc = idesc_f16(BF16, false, true, 128, kD);  // dV (TS), dK (SS)
        constexpr uint32_t kIdDQ = idesc_f16(BF16, true, true, 128, kD);    // dQ: both MN-major
        const uint64_t k_kmaj = smem_desc_sw128(smem_u32(smem + kOffK), 16, 1024);
        const uint64_t v_kmaj = smem_desc_sw128(smem_u32(smem + kOffV), 16, 1024);
        const uint64_t k_mnmaj = smem_desc_sw128(smem_u32(smem + kOffK), kBlock, 1024);
        const uint64_t ps_kmaj = smem_desc_sw128(smem_u32(smem + kOffPS), 16, 1024);
        const uint64_t ps_mnmaj = smem_desc_sw128(smem_u32(smem + kOffPS), kBlock, 1024);
        const uint32_t aQ0 = smem_u32(smem + kOffQ), aDO0 = smem_u32(smem + kOffDO);
        // S^T or dP^T: K = 64 head-dim elements, one column block
        auto issue_scores = [&](uint32_t d_col, uint64_t a_desc, uint32_t b_base) {
          const uint64_t bd = smem_desc_sw128(b_base, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            mma_f16_ss(tmem + d_col, a_desc + kstep_kmajor(kk), bd + kstep_kmajor(kk), kIdS, kk > 0 ? 1u : 0u);
        };
        bool ok = wait_bar(&bars->kv_full, 0, abort_flag, p.status) &&
                  wait_bar(&bars->qd_full[0], 0, abort_flag, p.status);
        if (ok) {
          tc_fence_after();
          if (chain_x) {
            issue_scores(kColX, k_kmaj, aQ0);
            mma_commit(&bars->s_full);
          } else {
            issue_scores(kColY, v_kmaj, aDO0);
            mma_commit(&bars->dp_full);
          }
        }
        if (chain_x) {
          for (int t = 0; ok && t < T; ++t) {
            const int s = t % kStages;
            const uint32_t ph = t & 1;
            // dV += P^T dO_t: A = P^T in tensor memory, B = dO_t MN-major (N = 64)
            if (!(ok = wait_bar(&bars->p_full, ph, abort_flag, p.status))) break;
            tc_fence_after();
            {
              const uint64_t bd = smem_desc_sw128(aDO0 + s * kTile, kBlock, 1024);
#pragma unroll
              for (int kk = 0; kk < kT / 16; ++kk)
                mma_f16_ts(tmem + kColDV, tmem + kColX + (kk / 4) * 64 + (kk % 4) * 8, bd + kstep_mnmajor(kk), kIdAcc,
                           (t > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&bars->dv_done);
            mma_commit(&bars->qd_empty[s]);
            if (t + 1 < T) {
              const int s1 = (t + 1) % kStages;
              if (!(ok = wait_bar(&bars->qd_full[s1], ((t + 1) / kStages) & 1, abort_flag, p.status))) break;
              if (!(ok = wait_bar(&bars->dv_done, ph, abort_flag, p.status))) break;
              tc_fence_after();
              issue_scores(kColX, k_kmaj, aQ0 + s1 * kTile);
              mma_commit(&bars->s_full);
            }
          }
        } else {
          for (int t = 0; ok && t < T; ++t) {
            const int s = t % kStages;
            const uint32_t ph = t & 1;
            if (t + 1 < T) {
              const int s1 = (t + 1) % kStages;
              if (!(ok = wait_bar(&bars->qd_full[s1], ((t + 1) / kStages) & 1, abort_flag, p.status))) break;
              if (!(ok = wait_bar(&bars->dp_free, ph, abort_flag, p.status))) break;
              tc_fence_after();
              issue_scores(kColY, v_kmaj, aDO0 + s1 * kTile);
              mma_commit(&bars->dp_full);
            }
            if (!(ok = wait_bar(&bars->ds_full, ph, abort_flag, p.status))) break;
            if (t > 0 && !(ok = wait_bar(&bars->dq_free, (t - 1) & 1, abort_flag, p.status))) break;
            tc_fence_after();
            // dQ(t) = dS K: A = dS^T read MN-major (M = 128 queries), B = K MN-major (N = 64)
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk)
              mma_f16_ss(tmem + kColQ, ps_mnmaj + kstep_mnmajor(kk), k_mnmaj + kstep_mnmajor(kk), kIdDQ,
                         kk > 0 ? 1u : 0u);
            mma_commit(&bars->dq_full);
            // dK += dS^T Q_t: the last reader of dS^T(t) and of Q_t
            {
              const uint64_t bd = smem_desc_sw128(aQ0 + s * kTile, kBlock, 1024);
#pragma unroll
              for (int kk = 0; kk < kT / 16; ++kk)
                mma_f16_ss(tmem + kColDK, ps_kmaj + kstep_kmajor(kk), bd + kstep_mnmajor(kk), kIdAcc,
                           (t > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&bars->dk_done);
            mma_commit(&bars->qd_empty[s]);
          }
        }
        mma_commit(&bars->acc_done);
        int dummy = 0;
        bounded_wait(&bars->acc_done, 0, reinterpret_cast<volatile int*>(&dummy), p.status, kStatusTimeoutDrain);
      }
      __syncwarp();
    }
  } else {
    // ================================================================ compute warpgroups
    regs_inc<kRegsCompute>();
    const int wg = warp / 4;
    const int kl = (warp % 4) * 32 + lane;  // key row (TMEM lane of S^T / dP^T)
    const int key = k0 + kl;
    const uint32_t lane_off = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t colX = tmem + lane_off + kColX + wg * 64;
    const uint32_t colY = tmem + lane_off + kColY + wg * 64;
    const float lam = p.scale_log2;
    float x[64];

    auto phase_p = [&](int t) -> bool {
      const int s = t % kStages;
      int h, q0;
      block_coords(t, h, q0);
      (void)h;
      const int c0 = q0 + wg * 64;
      const bool ok = wait_bar(&bars->s_full, t & 1, abort_flag, p.status) &&
                      wait_bar(&bars->qd_full[s], (t / kStages) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) return false;
      tc_fence_after();
      tmem_ld32(colX, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      tmem_ld32(colX + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      tmem_wait_ld();
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      const float4* st_l = reinterpret_cast<const float4*>(stats + s * 2 * kT + wg * 64);
      const bool need_mask = (k0 + kT > p.Sk) || (CAUSAL && (k0 + kT - 1 > c0 + p.delta));
      const int first_c = (key >= p.Sk) ? 64 : (CAUSAL ? key - p.delta - c0 : 0);
      const float2 lam2 = make_float2(lam, lam);
      if (!need_mask) {  // block-uniform: every block but the diagonal and ragged ones
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 l4 = st_l[c4];
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
          const float4 l4 = st_l[c4];
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
      {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack2<BF16>(x[2 * i], x[2 * i + 1]);
        tmem_st16(colX, pk);
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack2<BF16>(x[32 + 2 * i], x[32 + 2 * i + 1]);
        tmem_st16(colX + 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
      return true;
    };

    auto phase_ds = [&](int t) -> bool {
      const int s = t % kStages;
      bool ok = wait_bar(&bars->dp_full, t & 1, abort_flag, p.status);
      if (t > 0) ok = ok && wait_bar(&bars->dk_done, (t - 1) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) return false;
      tc_fence_after();
      const float4* st_d = reinterpret_cast<const float4*>(stats + s * 2 * kT + kT + wg * 64);
      uint8_t* row = smem + kOffPS + wg * kBlock + kl * 128;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t w[32];
        tmem_ld32(colY + hf * 32, w);
        tmem_wait_ld();
        reg_fence32(w);
        uint32_t pk[16];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 d4 = st_d[hf * 8 + c4];
          const int cb = hf * 32 + 4 * c4;
          const float2 a = fmul2(make_float2(x[cb], x[cb + 1]),
                                 fadd2(make_float2(__uint_as_float(w[4 * c4]), __uint_as_float(w[4 * c4 + 1])),
                                       make_float2(-d4.x, -d4.y)));
          const float2 b2 = fmul2(make_float2(x[cb + 2], x[cb + 3]),
                                  fadd2(make_float2(__uint_as_float(w[4 * c4 + 2]), __uint_as_float(w[4 * c4 + 3])),
                                        make_float2(-d4.z, -d4.w)));
          pk[2 * c4] = pack2<BF16>(a.x, a.y);
          pk[2 * c4 + 1] = pack2<BF16>(b2.x, b2.y);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int chunk = hf * 4 + c;
          *reinterpret_cast<uint4*>(row + ((chunk ^ (kl & 7)) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->dp_free);  // dP^T(t) is in registers: dP^T(t+1) may follow
      fence_proxy_async_smem();
      mbar_arrive(&bars->ds_full);
      return true;
    };

    bool ok = T > 0 && phase_p(0);
    for (int t = 0; ok && t < T; ++t) {
      if (!(ok = phase_ds(t))) break;
      if (t + 1 < T && !(ok = phase_p(t + 1))) break;
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
    // Sk are not written).  A thread storing its own 256-byte row to global
    // memory instead touches one cache line per lane and store instruction.
    uint8_t* stage = smem + (wg ? kOffK : kOffV) + kl * 128;
#pragma unroll 1
    for (int c = 0; c < kD / 32; ++c) {
      uint32_t w[32];
      if (have) {
        tmem_ld32(tmem + lane_off + (wg ? kColDK : kColDV) + c * 32, w);
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
      for (int cb = 0; cb < kD / 64; ++cb)
        tma_store_3d(wg ? &tmap_dk : &tmap_dv, smem + (wg ? kOffK : kOffV) + cb * kBlock, cb * 64, k0, bkv);
      bulk_commit_group();
      bulk_wait_group_read0();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarpX) tmem_dealloc(tmem, 512);
}

// D[row] = sum_t dO[row,t] * O[row,t] (fp32) and a zeroed accumulator row;
// DH / 8 threads per row, 8 elements (16 bytes) each.
template <int DH, bool BF16>
__global__ void __launch_bounds__(256) bwd_atomic_prep_kernel(const uint16_t* __restrict__ o,
                                                              const uint16_t* __restrict__ dout,
                                                              float* __restrict__ Dvec, float* __restrict__ dq_acc,
                                                              long long n_rows) {
  constexpr int kTpr = DH / 8;  // threads per row
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long r = tid / kTpr;
  const int part = static_cast<int>(tid % kTpr);
  float acc = 0.f;
  if (r < n_rows) {
    const uint4 a = *reinterpret_cast<const uint4*>(o + r * DH + part * 8);
    const uint4 c = *reinterpret_cast<const uint4*>(dout + r * DH + part * 8);
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
    float4* z = reinterpret_cast<float4*>(dq_acc + r * DH + part * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (r < n_rows && part == 0) Dvec[r] = acc;
}

// dQ = tau * accumulator in the input dtype; 8 elements per thread.
template <bool BF16>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq,
                                                             float scale, long long n8) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
  const float4 c = reinterpret_cast<const float4*>(acc)[2 * i + 1];
  reinterpret_cast<uint4*>(dq)[i] =
      make_uint4(pack2<BF16>(a.x * scale, a.y * scale), pack2<BF16>(a.z * scale, a.w * scale),
                 pack2<BF16>(c.x * scale, c.y * scale), pack2<BF16>(c.z * scale, c.w * scale));
}

// KV heads per scheduling group, counted in the Q, dO and fp32 accumulator
// rows a group re-reads.  The budget is 256 MB -- larger than L2 -- because
// for this kernel balancing heavy and light causal key tiles across more
// heads outweighs keeping a group's rows resident: measured (launch-by-launch
// alternation) against a 48 MB budget, GQA causal 0.842 -> 0.703 ms at 16 KV
// heads per group, causal [4,16,8192,128] 2.77 -> 2.65 ms at 32.
int head_group_atomic(long long per_head_bytes, long long heads) {
  long long hg = (256LL << 20) / (per_head_bytes > 0 ? per_head_bytes : 1);
  if (hg < 1) hg = 1;
  return balanced_head_group(hg, heads, 1);
}

template <int DH, bool BF16, bool CAUSAL>
int launch_atomic_t(const BackwardArgs& a) {
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
  if (!make_tmap_3d(&tq, a.q, BF16, DH, a.Sq, static_cast<long long>(a.B) * a.H, kT) ||
      !make_tmap_3d(&tdo, a.dout, BF16, DH, a.Sq, static_cast<long long>(a.B) * a.H, kT) ||
      !make_tmap_3d(&tk, a.k, BF16, DH, a.Sk, static_cast<long long>(a.B) * a.Hkv, kT) ||
      !make_tmap_3d(&tv, a.v, BF16, DH, a.Sk, static_cast<long long>(a.B) * a.Hkv, kT) ||
      !make_tmap_3d(&tdk, a.dk, BF16, DH, a.Sk, static_cast<long long>(a.B) * a.Hkv, kT) ||
      !make_tmap_3d(&tdv, a.dv, BF16, DH, a.Sk, static_cast<long long>(a.B) * a.Hkv, kT))
    return -1;
  if (DH == 64 && !make_tmap_3d_f32(&tdq, a.dq_acc, DH, a.Sq, static_cast<long long>(a.B) * a.H, 32, 32))
    return -1;
  const long long n_rows = static_cast<long long>(a.B) * a.H * a.Sq;
  {
    const long long blocks = (n_rows * (DH / 8) + 255) / 256;
    if (blocks > 0x7FFFFFFFLL) return -1;
    bwd_atomic_prep_kernel<DH, BF16><<<static_cast<unsigned>(blocks), 256, 0, a.stream>>>(
        static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dout), a.Dvec, a.dq_acc, n_rows);
  }
  const int smem_bytes = DH == 64 ? d64::kSmemBytes : kSmemBytes;
  static std::atomic<unsigned long long> attr_done{0};  // per instantiation
  const bool attr_ok = DH == 64 ? set_smem_limit_once(bwd_atomic64_kernel<BF16, CAUSAL>, smem_bytes, attr_done)
                                : set_smem_limit_once(bwd_atomic_kernel<BF16, CAUSAL>, smem_bytes, attr_done);
  if (!attr_ok) return -1;
  AtomicParams p;
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
  p.n_ktiles = (a.Sk + kT - 1) / kT;
  p.n_qtiles = (a.Sq + kT - 1) / kT;
  p.delta = a.Sk - a.Sq;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.status = a.status;
  p.head_group = head_group_atomic(static_cast<long long>(p.g) * a.Sq * DH * 8, static_cast<long long>(a.B) * a.Hkv);
  const long long grid = static_cast<long long>(a.B) * a.Hkv * p.n_ktiles;
  if (grid > 0x7FFFFFFFLL) return -1;
  if constexpr (DH == 64)
    bwd_atomic64_kernel<BF16, CAUSAL><<<static_cast<unsigned>(grid), kThreads, smem_bytes, a.stream>>>(tq, tk, tv, tdo,
                                                                                                      tdq, tdk, tdv, p);
  else
    bwd_atomic_kernel<BF16, CAUSAL><<<static_cast<unsigned>(grid), kThreads, smem_bytes, a.stream>>>(tq, tk, tv, tdo,
                                                                                                    tdk, tdv, p);
  {
    const long long n8 = n_rows * (DH / 8);
    const long long blocks = (n8 + 255) / 256;
    if (blocks > 0x7FFFFFFFLL) return -1;
    bwd_dq_convert_kernel<BF16><<<static_cast<unsigned>(blocks), 256, 0, a.stream>>>(
        a.dq_acc, static_cast<uint16_t*>(a.dq), a.scale, n8);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_backward_atomic(const BackwardArgs& a) {
  if (!a.dq_acc) return -1;
  if (a.d == 128) {
    if (a.bf16) return a.causal ? launch_atomic_t<128, true, true>(a) : launch_atomic_t<128, true, false>(a);
    return a.causal ? launch_atomic_t<128, false, true>(a) : launch_atomic_t<128, false, false>(a);
  }
  if (a.d != 64) return -1;
  if (a.bf16) return a.causal ? launch_atomic_t<64, true, true>(a) : launch_atomic_t<64, true, false>(a);
  return a.causal ? launch_atomic_t<64, false, true>(a) : launch_atomic_t<64, false, false>(a);
}

}  // namespace gbattn
