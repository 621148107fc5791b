// prefill_pair.cu -- non-causal exact attention forward, d = 128, on a tcgen05
// CTA pair (cta_group::2): two CTAs of a cluster share every K/V tile.
//
// A cluster of two CTAs owns four 128-row query tiles of one (batch, query
// head): rank r holds tile H = rows [512u + 128r, +128) and tile L = rows
// [512u + 256 + 128r, +128).  Rank 0 issues every MMA for the pair as an
// M = 256 product (M4.6 "FlashAttention-3/4 Hardware Pipelines" 0x08, the
// 2-CTA mode of the non-causal d = 128 forward):
//   S_X  = Q_X K^T    A = Q_X (each CTA its own 128 rows, K-major)
//                     B = K tile, N = 128 keys: rank r supplies keys [64r, 64r+64)
//   O_X += P_X V      A = P_X (each CTA its own rows, K-major, shared memory)
//                     B = V tile, N = d = 128: rank r supplies d columns [64r, 64r+64)
// Each CTA's tensor memory receives its own 128 rows of S and O over all
// columns, so the softmax, correction and epilogue are those of the one-CTA
// forward (prefill_fwd.cu) on local data.  What the pair changes:
//   - each CTA loads half of every K and V tile (16 KiB instead of 32 KiB),
//     and the tensor core of each SM reads half of every B operand from its
//     own shared memory;
//   - one thread issues the MMAs of both SMs (half the issue work per SM);
//   - the freed shared memory holds three 64-key P blocks per query tile
//     instead of two: P(j) block b goes to block slot (2j + b) mod 3, so
//     P(j+1) waits only for the first half of P.V(j) (one wait per key tile,
//     before its first block), never for the whole of it.  The pair's
//     handshakes cross the cluster (about 570 cycles one way, measured).
//
// Cross-CTA protocol (cluster-scope mbarriers; every wait bounded):
//   loads      each CTA's TMA lane loads its Q tiles and K/V halves and
//              completes its own q_full / kv_full; rank 1's warp 8 forwards
//              every completion to rank 0's q_peer / kv_peer (remote arrive)
//   S ready    rank 0 commits to s_full in both CTAs (multicast commit)
//   S copied   each softmax warp arrives once on rank 0's s_free (4 + 4)
//   P written  each softmax warp arrives once on rank 0's p_full (4 + 4)
//   P.V done   multicast commits to pblk_free (per P block slot) / o_full
//   slot free  multicast commits to kv_empty of both CTAs
//   stagger    tile H's softmax warps of both CTAs arrive once, after their
//              first S copy, on rank 0's stagger; tile L's issuer waits for
//              it before QK_L(0), so the tiles' softmax chains run apart
// Tensor memory is allocated and freed pair-collectively (warp 8 of each
// CTA); the kernel ends with two cluster barriers around the free.
//
// Online softmax, rescale threshold and the epilogue are those of
// prefill_fwd.cu; the correction of O (rare with threshold 8) waits for the
// whole of P.V(j-1) only in warps where a row moved its reference.
#include <cuda_runtime.h>

#include "gbattn_internal.h"
#include "gbattn_ptx.cuh"

namespace gbattn {
namespace {

constexpr int kBM = 128;  // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kD = 128;   // head dim
constexpr int kThreads = 384;
constexpr int kSoftmaxRegs = 224;
constexpr int kControlRegs = 56;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * 168, "register split");
constexpr int kMmaWarpH = 8;   // rank 0: tile H issuer; rank 1: completion forwarder
constexpr int kLoadWarp = 9;
constexpr int kMmaWarpL = 10;  // rank 0: tile L issuer; rank 1: waits for the last commits
constexpr float kRescaleThreshold = 8.0f;  // log2 units (fp16/bf16 row of M4.6 0x09 table)

constexpr int kTileBytes = kBM * kD * 2;  // 32 KiB: one 128 x 128 16-bit tile
constexpr int kBlockBytes = kBM * 128;    // 16 KiB: 128 rows x 128 bytes (one swizzle column block)
constexpr int kHalfBytes = 16384;         // this CTA's half of a K or V tile
constexpr int kKBlockBytes = 64 * 128;    // 8 KiB: 64 key rows x 128 bytes
constexpr int kStages = 4;                // K/V half-tile ring slots
constexpr int kPSlots = 3;                // 64-key P block slots per query tile
constexpr int kQOff = 0;
constexpr int kPOff = 2 * kTileBytes;
constexpr int kRingOff = kPOff + 2 * kPSlots * kBlockBytes;
constexpr int kBarOff = kRingOff + kStages * kHalfBytes;
constexpr int kSmemBytes = 1024 + kBarOff + 512;  // + alignment slack + barriers
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
  void* o;
  float* lse;
  int B, H, Hkv, Sq, Sk, g;
  int n_quads;     // 512-row query units per (batch, head)
  int head_group;  // (batch, head) pairs per L2 scheduling group
  float scale_log2;
  int* status;
  int wave;                       // CTAs resident at once (one per SM)
  unsigned long long* timeline;   // optional per-CTA records, or null
};

struct __align__(8) Barriers {
  uint64_t q_full;
  uint64_t q_peer;  // rank 0: rank 1's Q tiles landed
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t kv_peer[kStages];  // rank 0: rank 1's half of the item landed
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t pblk_free[2][kPSlots];  // the P.V half reading this P block slot is complete
  uint64_t o_full[2];
  uint64_t mma_done[2];
  uint64_t stagger;  // rank 0: tile H of both CTAs has read its first S
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Barriers) <= 512, "barrier block");

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Position of K_j / V_j in the load order K_0, K_1, V_0, K_2, V_1, ...,
// K_{n-1}, V_{n-2}, V_{n-1} (n key tiles).
__device__ __forceinline__ int item_of_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int item_of_v(int j, int n) { return j <= n - 2 ? 2 * j + 2 : 2 * n - 1; }

template <bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_o,
                        const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + kQOff;
  uint8_t* sP = smem + kPOff;
  uint8_t* sRing = smem + kRingOff;
  Barriers* bars = reinterpret_cast<Barriers*>(smem + kBarOff);
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  unsigned long long t_start = 0;
  if (p.timeline != nullptr && threadIdx.x == 0) t_start = global_timer_ns();

  // ---- work unit (one per cluster), in groups of p.head_group (batch, head)
  // pairs whose K/V stay resident in L2, heads fastest.
  const int unit = static_cast<int>(blockIdx.x >> 1);
  const int BH = p.B * p.H;
  const int group = unit / (p.head_group * p.n_quads);
  const int heads_here = min(p.head_group, BH - group * p.head_group);
  const int r_in = unit - group * p.head_group * p.n_quads;
  const int bh = group * p.head_group + r_in % heads_here;
  const int quad = r_in / heads_here;
  const int b = bh / p.H;
  const int h = bh % p.H;
  const int kvh = h / p.g;
  const int q0_h = quad * 4 * kBM + static_cast<int>(rank) * kBM;
  const int q0_l = q0_h + 2 * kBM;
  const int nt = ceil_div(p.Sk, kBN);  // every tile of the pair visits every key tile
  const int n_items = 2 * nt;

  // ---- setup
  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_peer, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 2);  // one multicast commit from each issuer
      mbar_init(&bars->kv_peer[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars->s_full[x], 1);
      mbar_init(&bars->s_free[x], 8);  // one arrival per softmax warp of either CTA
      mbar_init(&bars->p_full[x], 8);
      for (int sl = 0; sl < kPSlots; ++sl) mbar_init(&bars->pblk_free[x][sl], 1);
      mbar_init(&bars->o_full[x], 1);
      mbar_init(&bars->mma_done[x], 1);
    }
    mbar_init(&bars->stagger, 8);  // one arrival per tile-H softmax warp of either CTA
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  if (warp == kMmaWarpH) {
    tmem_alloc_pair(&bars->tmem_base, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp >= 8) {
    // ---- control warpgroup
    regs_dec<kControlRegs>();
    if (warp == kLoadWarp) {
      // ================================================================ loader (both CTAs)
      if (lane == 0) {
        const uint64_t keep = policy_evict_last();   // K/V: re-read by other clusters
        const uint64_t once = policy_evict_first();  // Q: read by this CTA only
        mbar_arrive_expect_tx(&bars->q_full, 2 * kTileBytes);
        for (int x = 0; x < 2; ++x)
          for (int cb = 0; cb < 2; ++cb)
            tma_load_3d(sQ + x * kTileBytes + cb * kBlockBytes, &tmap_q, &bars->q_full, cb * 64, x ? q0_l : q0_h,
                        b * p.H + h, once);
        {  // this CTA's Q rows of the cluster unit one wave ahead into L2
          const int ahead = unit + p.wave / 2;
          if (ahead < static_cast<int>(gridDim.x >> 1)) {
            const int ga = ahead / (p.head_group * p.n_quads);
            const int heads_a = min(p.head_group, BH - ga * p.head_group);
            const int ra = ahead - ga * p.head_group * p.n_quads;
            const int bh_a = ga * p.head_group + ra % heads_a;
            const int qa = (ra / heads_a) * 4 * kBM + static_cast<int>(rank) * kBM;
            for (int x = 0; x < 2; ++x)
              if (qa + 2 * x * kBM < p.Sq)
                for (int cb = 0; cb < 2; ++cb) tma_prefetch_l2_3d(&tmap_q, cb * 64, qa + 2 * x * kBM, bh_a);
          }
        }
        int issued = 0;
        for (int it = 0; it < n_items; ++it) {
          const int st = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!bounded_wait(&bars->kv_empty[st], ph ^ 1, abort_flag, p.status, kStatusTimeoutLoad)) break;
          bool is_v;
          int jt;
          if (it == 0) {
            is_v = false, jt = 0;
          } else if (it & 1) {
            if (it == n_items - 1) is_v = true, jt = nt - 1;
            else is_v = false, jt = (it + 1) / 2;
          } else {
            is_v = true, jt = (it - 2) / 2;
          }
          mbar_arrive_expect_tx(&bars->kv_full[st], kHalfBytes);
          uint8_t* dst = sRing + st * kHalfBytes;
          if (is_v) {  // d columns [64 rank, 64 rank + 64) of all 128 keys (MN-major B of P.V)
            tma_load_3d(dst, &tmap_v, &bars->kv_full[st], 64 * static_cast<int>(rank), jt * kBN, b * p.Hkv + kvh,
                        keep);
          } else {  // keys [64 rank, 64 rank + 64) of the tile, both d column blocks (K-major B of QK)
            for (int cb = 0; cb < 2; ++cb)
              tma_load_3d(dst + cb * kKBlockBytes, &tmap_k, &bars->kv_full[st], cb * 64,
                          jt * kBN + 64 * static_cast<int>(rank), b * p.Hkv + kvh, keep);
          }
          issued = it + 1;
        }
        // Drain: every copy this thread issued must have landed before exit.
        bounded_wait(&bars->q_full, 0, abort_flag, p.status, kStatusTimeoutDrain);
        for (int it = max(0, issued - kStages); it < issued; ++it) {
          int dummy = 0;
          bounded_wait(&bars->kv_full[it % kStages], (it / kStages) & 1, reinterpret_cast<volatile int*>(&dummy),
                       p.status, kStatusTimeoutDrain);
        }
      }
      __syncwarp();
    } else if (!leader) {
      if (warp == kMmaWarpH && lane == 0) {
        // ================================================================ forwarder (rank 1)
        // Rank 0 may read this CTA's operands only once they have landed here.
        if (bounded_wait(&bars->q_full, 0, abort_flag, p.status, kStatusTimeoutMma)) {
          mbar_arrive_cluster_smem_release(mapa_shared(&bars->q_peer, 0));
          for (int it = 0; it < n_items; ++it) {
            const int st = it % kStages;
            if (!bounded_wait(&bars->kv_full[st], (it / kStages) & 1, abort_flag, p.status, kStatusTimeoutMma))
              break;
            mbar_arrive_cluster_smem_release(mapa_shared(&bars->kv_peer[st], 0));
          }
        }
      } else if (warp == kMmaWarpL && lane == 0) {
        // The last multicast commits of rank 0 land in this CTA's barriers
        // before it may exit.
        for (int x = 0; x < 2; ++x) {
          int dummy = 0;
          bounded_wait(&bars->mma_done[x], 0, reinterpret_cast<volatile int*>(&dummy), p.status,
                       kStatusTimeoutDrain);
        }
      }
      __syncwarp();
    } else if (warp == kMmaWarpH || warp == kMmaWarpL) {
      // ================================================================ MMA issuers (rank 0)
      if (lane == 0) {
        const int x = (warp == kMmaWarpH) ? 0 : 1;
        constexpr uint32_t kIdescQK = idesc_f16(BF16, false, false, 2 * kBM, kBN);
        constexpr uint32_t kIdescPV = idesc_f16(BF16, false, true, 2 * kBM, kD);
        const uint32_t ring_addr = smem_u32(sRing);
        const uint32_t s_col = tmem + x * kBN;
        const uint32_t o_col = tmem + 2 * kBN + x * kD;
        const uint64_t q_desc = smem_desc_sw128(smem_u32(sQ + x * kTileBytes), 16, 1024);
        const uint32_t p_base = smem_u32(sP + x * kPSlots * kBlockBytes);
        // Both halves of an item must have landed (own kv_full, forwarded kv_peer).
        auto wait_item = [&](int item) -> int {
          const int st = item % kStages;
          const uint32_t par = (item / kStages) & 1;
          if (!bounded_wait(&bars->kv_full[st], par, abort_flag, p.status, kStatusTimeoutMma)) return -1;
          if (!bounded_wait_cluster(&bars->kv_peer[st], par, abort_flag, p.status, kStatusTimeoutMma)) return -1;
          return st;
        };
        // K-step kk covers d [16 kk, 16 kk + 16): A (Q) column blocks are
        // 16 KiB apart, B (this CTA's 64 keys) column blocks 8 KiB apart.
        auto issue_qk = [&](int st) {
          const uint64_t kd = smem_desc_sw128(ring_addr + st * kHalfBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint64_t aoff = ((kk / 4) * kBlockBytes + (kk % 4) * 32) >> 4;
            const uint64_t boff = ((kk / 4) * kKBlockBytes + (kk % 4) * 32) >> 4;
            mma_pair_f16_ss(s_col, q_desc + aoff, kd + boff, kIdescQK, kk > 0 ? 1u : 0u);
          }
        };
        // P.V over keys [64 half, 64 half + 64) of key tile j: P block slot
        // (2j + half) mod 3; the V half is one MN-major column block, 16 key
        // rows = 2 KiB per K-step.
        auto issue_pv_half = [&](int st, int j, int half, bool accumulate) {
          const uint64_t vd = smem_desc_sw128(ring_addr + st * kHalfBytes, kHalfBytes, 1024);
          const uint64_t pd = smem_desc_sw128(p_base + ((2 * j + half) % kPSlots) * kBlockBytes, 16, 1024);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = half * 4 + k4;
            mma_pair_f16_ss(o_col, pd + ((k4 * 32) >> 4), vd + ((kk * 2048) >> 4), kIdescPV,
                            (accumulate || kk > 0) ? 1u : 0u);
          }
        };
        bool ok = bounded_wait(&bars->q_full, 0, abort_flag, p.status, kStatusTimeoutMma) &&
                  bounded_wait_cluster(&bars->q_peer, 0, abort_flag, p.status, kStatusTimeoutMma);
        // Tile L's first QK waits until tile H has read S_H(0) in both CTAs, so
        // the two tiles' softmax chains run staggered instead of in lockstep.
        if (ok && x == 1) ok = bounded_wait_cluster(&bars->stagger, 0, abort_flag, p.status, kStatusTimeoutMma);
        if (ok) {
          const int st = wait_item(item_of_k(0));
          ok = st >= 0;
          if (ok) {
            tc_fence_after();
            issue_qk(st);
            mma_commit_pair(&bars->s_full[x]);
            mma_commit_pair(&bars->kv_empty[st]);
          }
        }
        for (int j = 0; ok && j < nt; ++j) {
          // QK_X(j+1) once both CTAs' softmax threads hold S_X(j) in registers
          if (j + 1 < nt) {
            const int st = wait_item(item_of_k(j + 1));
            ok = st >= 0;
            if (!ok) break;
            if (!(ok = bounded_wait_cluster(&bars->s_free[x], j & 1, abort_flag, p.status, kStatusTimeoutMma)))
              break;
            tc_fence_after();
            issue_qk(st);
            mma_commit_pair(&bars->s_full[x]);
            mma_commit_pair(&bars->kv_empty[st]);
          }
          // PV_X(j) once both CTAs have written P_X(j) (and corrected O_X)
          {
            const int st = wait_item(item_of_v(j, nt));
            ok = st >= 0;
            if (!ok) break;
            if (!(ok = bounded_wait_cluster(&bars->p_full[x], j & 1, abort_flag, p.status, kStatusTimeoutMma)))
              break;
            tc_fence_after();
            issue_pv_half(st, j, 0, j > 0);
            mma_commit_pair(&bars->pblk_free[x][(2 * j) % kPSlots]);
            issue_pv_half(st, j, 1, true);
            mma_commit_pair(&bars->pblk_free[x][(2 * j + 1) % kPSlots]);
            if (j == nt - 1) mma_commit_pair(&bars->o_full[x]);
            mma_commit_pair(&bars->kv_empty[st]);
          }
        }
        // Every MMA this thread issued must complete before TMEM is released.
        mma_commit_pair(&bars->mma_done[x]);
        int dummy = 0;
        bounded_wait(&bars->mma_done[x], 0, reinterpret_cast<volatile int*>(&dummy), p.status, kStatusTimeoutDrain);
      }
      __syncwarp();
    }
  } else {
    // ---- softmax warpgroups (both CTAs, on their own rows)
    regs_inc<kSoftmaxRegs>();
    const int x = warp / 4;   // 0 = tile H, 1 = tile L
    const int wq = warp % 4;  // TMEM lane quarter owned by this warp
    const int row = wq * 32 + lane;
    const int q0x = x ? q0_l : q0_h;
    const int q_row = q0x + row;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_tmem = tmem + lane_off + x * kBN;
    const uint32_t o_tmem = tmem + lane_off + 2 * kBN + x * kD;
    // Rank 0's s_free / p_full (local address on rank 0, remote on rank 1).
    const uint32_t s_free_addr = mapa_shared(&bars->s_free[x], 0);
    const uint32_t p_full_addr = mapa_shared(&bars->p_full[x], 0);
    const uint32_t stagger_addr = mapa_shared(&bars->stagger, 0);
    // This row of P_X in shared memory: block slots of 64 keys in 128-byte
    // rows; 16-byte chunk c of the row sits at chunk c ^ (row % 8).
    uint8_t* p_row = sP + x * kPSlots * kBlockBytes + row * 128;
    const float lam = p.scale_log2;
    float r = -INFINITY;  // retained reference, raw score units
    float l = 0.f;
    bool ok = true;

    for (int j = 0; j < nt; ++j) {
      ok = bounded_wait_cluster(&bars->s_full[x], j & 1, abort_flag, p.status, kStatusTimeoutSoftmax);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // ---- S row -> registers, then S_X of this CTA is free; a tile without
      // a key tail also gets each 32-column block's maximum from the loads
      const int k0 = j * kBN;
      const bool key_tail = k0 + kBN > p.Sk;
      uint32_t u[kBN];
      float mq[kBN / 32];
      if (key_tail) {
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c)
          tmem_ld32(s_tmem + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&u[c * 32]));
      } else {
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c)
          tmem_ld32_max(s_tmem + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&u[c * 32]), mq[c]);
      }
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&u[c * 32]));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {  // rank 0: local arrive; rank 1: shared-memory release + relaxed remote arrive
        if (leader) mbar_arrive(&bars->s_free[x]);
        else mbar_arrive_cluster_smem_release(s_free_addr);
        if (x == 0 && j == 0) {
          if (leader) mbar_arrive(&bars->stagger);
          else mbar_arrive_cluster_smem_release(stagger_addr);
        }
      }
      float* s = reinterpret_cast<float*>(u);
      float mx;
      if (key_tail) {
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (k0 + c >= p.Sk) s[c] = -INFINITY;
        // ---- row maximum: eight independent three-input max chains
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = s[i];
#pragma unroll
        for (int c = 8; c < kBN; c += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], s[c + i], s[c + 8 + i < kBN ? c + 8 + i : c + i]);
        mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
      } else {
        mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      }
      float gamma = 1.f;
      if (j == 0) {
        r = mx;
      } else {
        const float cand = fmaxf(r, mx);
        if ((cand - r) * lam > kRescaleThreshold) {  // false when both are -inf
          gamma = ex2_approx((r - cand) * lam);
          r = cand;
        }
      }
      l *= gamma;
      // ---- P = 2^(lambda*s - lambda*r), row sum, pack to 16 bits, store the
      // row of P_X(j): block b (n = 2j + b) into slot n mod 3 once the P.V
      // halves that read the slots' previous blocks are complete; before the
      // last block, O is corrected once P.V_X(j-1) is complete.
      const float rs = (r == -INFINITY) ? 0.f : r * lam;
      const float2 lam2 = make_float2(lam, lam);
      const float2 nrs2 = make_float2(-rs, -rs);
      float2 sum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
#pragma unroll
      for (int blk = 0; blk < kBN / 64; ++blk) {
        uint32_t pk[32];
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {  // 16-byte chunks of 8 keys
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = blk * 64 + c8 * 8 + 2 * i;
            const float2 t = ex2_pair(ffma2(make_float2(s[c], s[c + 1]), lam2, nrs2), (blk * 8 + c8) * 4 + i);
            sum4[i] = fadd2(sum4[i], t);
            pk[c8 * 4 + i] = pack2<BF16>(t.x, t.y);
          }
        }
        if (blk == 0 && j >= 1) {
          // One wait per key tile: the first half of P.V_X(j-1) (block
          // n' = 2j - 2) complete implies every earlier P.V of the issuer
          // complete, so both slots P_X(j) goes to are free (block 0's slot
          // was last read by the second half of P.V_X(j-2), block 1's by the
          // first half of P.V_X(j-1)).  Measured 2.3 % faster than a wait
          // per block.
          const int np = 2 * j - 2;
          ok = bounded_wait_cluster(&bars->pblk_free[x][np % kPSlots], (np / kPSlots) & 1, abort_flag,
                                    p.status, kStatusTimeoutSoftmax);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
        }
        if (blk == kBN / 64 - 1 && j > 0 && __any_sync(0xffffffffu, gamma != 1.f)) {
          // correction: O_row *= gamma once P.V_X(j-1) (its second half,
          // block n' = 2j - 1) is complete; gamma = 1 rows unchanged
          const int np = 2 * j - 1;
          ok = bounded_wait_cluster(&bars->pblk_free[x][np % kPSlots], (np / kPSlots) & 1, abort_flag, p.status,
                                    kStatusTimeoutSoftmax);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < kD / 32; ++c) {
            uint32_t w32[32];
            tmem_ld32(o_tmem + c * 32, w32);
            tmem_wait_ld();
            reg_fence32(w32);
#pragma unroll
            for (int i = 0; i < 32; ++i) w32[i] = __float_as_uint(__uint_as_float(w32[i]) * gamma);
            tmem_st32(o_tmem + c * 32, w32);
          }
          tmem_wait_st();
        }
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)
          *reinterpret_cast<uint4*>(p_row + ((2 * j + blk) % kPSlots) * kBlockBytes + ((c8 ^ (row & 7)) << 4)) =
              make_uint4(pk[c8 * 4], pk[c8 * 4 + 1], pk[c8 * 4 + 2], pk[c8 * 4 + 3]);
      }
      if (!ok) break;
      const float2 s01 = fadd2(fadd2(sum4[0], sum4[1]), fadd2(sum4[2], sum4[3]));
      l += s01.x + s01.y;
      fence_proxy_async_smem();  // P stores -> visible to the tensor core (async proxy)
      tc_fence_before();         // O correction (tcgen05.st) ordered before the arrive
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&bars->p_full[x]);
        else mbar_arrive_cluster_smem_release(p_full_addr);
      }
    }

    // ---- epilogue: O = O / l, LSE
    if (q0x < p.Sq) {
      bool have_o = false;
      if (ok && nt > 0) {
        have_o = bounded_wait_cluster(&bars->o_full[x], 0, abort_flag, p.status, kStatusTimeoutSoftmax);
        have_o = __all_sync(0xffffffffu, have_o);
        tc_fence_after();
      }
      const bool row_ok = q_row < p.Sq;
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      // O_X is staged in Q_X (dead since the last QK_X completed), 128-byte
      // rows with 16-byte chunk c at chunk c ^ (row % 8), and written by one
      // TMA store per 64-column block (rows past Sq are not written).
      uint8_t* o_row = sQ + x * kTileBytes + row * 128;
#pragma unroll 1
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t w[32];
        if (have_o) {
          tmem_ld32(o_tmem + c * 32, w);
          tmem_wait_ld();
          reg_fence32(w);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2<BF16>(__uint_as_float(w[2 * i]) * inv, __uint_as_float(w[2 * i + 1]) * inv);
        uint8_t* blk = o_row + (c / 2) * kBlockBytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int ch = (c % 2) * 4 + k;
          *reinterpret_cast<uint4*>(blk + ((ch ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1 + x, kBM);
      if (wq == 0 && lane == 0) {
        for (int cb = 0; cb < 2; ++cb)
          tma_store_3d(&tmap_o, sQ + x * kTileBytes + cb * kBlockBytes, cb * 64, q0x, b * p.H + h);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
      if (row_ok && p.lse != nullptr) {
        const float lse = (l > 0.f) ? (r * lam + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        p.lse[(static_cast<size_t>(b) * p.H + h) * p.Sq + q_row] = lse;
      }
    }
  }

  // ---- teardown: every MMA of the pair complete (rank 0's issuers waited
  // for them, rank 1 for their last commits) before the pair frees TMEM
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  if (p.timeline != nullptr && threadIdx.x == 0) {
    // Timeline record of this CTA: start and end (%globaltimer ns), SM, unit.
    unsigned long long* rec = p.timeline + 4 * static_cast<size_t>(blockIdx.x);
    rec[0] = t_start;
    rec[1] = global_timer_ns();
    rec[2] = sm_id();
    rec[3] = static_cast<unsigned long long>(bh) << 32 | static_cast<unsigned>(quad);
  }
  if (warp == kMmaWarpH) tmem_dealloc_pair(tmem, 512);
  cluster_sync_all();
}

template <bool BF16>
int launch_pair_t(const PrefillArgs& a) {
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap_3d(&tq, a.q, BF16, kD, a.Sq, static_cast<long long>(a.B) * a.H, kBM) ||
      !make_tmap_3d(&to, a.o, BF16, kD, a.Sq, static_cast<long long>(a.B) * a.H, kBM) ||
      !make_tmap_3d(&tk, a.k, BF16, kD, a.Sk, static_cast<long long>(a.B) * a.Hkv, 64) ||
      !make_tmap_3d(&tv, a.v, BF16, kD, a.Sk, static_cast<long long>(a.B) * a.Hkv, kBN))
    return -1;
  auto kern = prefill_pair_kernel<BF16>;
  static std::atomic<unsigned long long> attr_done{0};  // per instantiation
  if (!set_smem_limit_once(kern, kSmemBytes, attr_done)) return -1;
  Params p{};
  p.o = a.o;
  p.lse = a.lse;
  p.B = a.B;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Sk = a.Sk;
  p.g = a.H / a.Hkv;
  p.n_quads = (a.Sq + 4 * kBM - 1) / (4 * kBM);
  {
    // Heads per scheduling group: about 48 MB of K/V in flight (L2 is 129 MB),
    // whole KV-head groups, groups of equal size (balanced_head_group).
    const long long kv_head_bytes = 4LL * a.Sk * kD;  // K and V, 16-bit
    long long kv_heads = (48LL << 20) / (kv_head_bytes > 0 ? kv_head_bytes : 1);
    if (kv_heads < 1) kv_heads = 1;
    p.head_group = balanced_head_group(kv_heads * p.g, static_cast<long long>(a.B) * a.H, p.g);
  }
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.status = a.status;
  p.wave = a.num_sms;
  const long long grid = 2LL * a.B * a.H * p.n_quads;
  if (grid > 0x7FFFFFFFLL) return -1;
  p.timeline = (a.timeline != nullptr && a.timeline_capacity >= grid) ? a.timeline : nullptr;
  kern<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, a.stream>>>(tq, tk, tv, to, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_prefill_pair(const PrefillArgs& a) {
  if (a.d != kD || a.causal) return -1;
  return a.bf16 ? launch_pair_t<true>(a) : launch_pair_t<false>(a);
}

}  // namespace gbattn
