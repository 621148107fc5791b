// prefill_fwd.cu -- exact attention forward on sm_103a: TMA-fed shared-memory
// ring, tcgen05 MMAs accumulating in tensor memory, warp-specialised roles.
//
// One CTA owns a pair of 128-row query tiles ("H" = rows [256p, 256p+128),
// "L" = the next 128 rows) of one (batch, query head) and streams every
// visible 128-key K/V tile of that head's KV head once for both query tiles
// (M4.4 0x03 Algorithm 1: query-tile owner; M4.6 0x08: two query tiles per
// CTA share each K/V tile).
//
// Tensor memory (512 columns, 128 lanes; lane = query row of the tile):
//   S_H  [  0,128)  fp32 scores of tile H      S_L  [128,256)  of tile L
//   O_H  [256,256+d)  unnormalised output      O_L  [256+d,256+2d)
//   d = 64 only: P_H [384,448), P_L [448,512)  16-bit P, keys (2c, 2c+1) in column c
// (the M4.6 0x07 capacity rule 2N + 2 d_v <= 512).
//
// Shared memory: Q_H, Q_L; d = 128: P_H, P_L (16-bit probabilities, K-major
// with the 128-byte swizzle, the A operand of the P.V MMA); a ring of K/V
// slots.
//
// Why P does not alias S: with P written over its S columns (the pages'
// FA4 map), QK(j+1) may only start after PV(j) has read P(j), so every
// tile's softmax sits on the critical path of the tensor pipe.  With P in a
// buffer of its own, QK_X(j+1) is issued as soon as the softmax threads have
// copied S_X(j) into registers.  At d = 128 tensor memory is full (S and O
// of both tiles), so P goes to shared memory and P.V reads both operands
// from there (8 KB per 16-key step for 16 KB of tensor work: balanced).  At
// d = 64 the 128 columns S and O leave free hold P for both tiles: the
// softmax writes P with tcgen05.st and P.V reads A from tensor memory (a TS
// MMA) and only V from shared memory.  Measured against P in shared memory
// at d = 64: 0.0575 -> 0.0498 ms.  The tensor pipe takes about as long for
// either form (48 and 45 cycles per 128x64x16 step); the shared-memory form
// adds the P stores, a proxy fence and 4 KB more operand reads per step.
//
// Warp roles (384 threads = three warpgroups):
//   warps 0-3   softmax + correction + epilogue of tile H (thread = one row)
//   warps 4-7   the same for tile L
//   warp  8     TMEM allocation; lane 0 issues tile H's MMAs and commits
//   warp  9     lane 0 issues every TMA copy
//   warp  10    lane 0 issues tile L's MMAs and commits
//   warp  11    idle
// Registers: launched at 168 per thread; the control warpgroup drops to 56
// and the two softmax warpgroups rise to 224 (2*128*224 + 128*56 = 384*168).
//
// Per tile X and key tile j (M4.6 0x08-0x09 roles, own protocol):
//   MMA X:     QK_X(0); then for j: [S_X(j) copied] QK_X(j+1);
//              [P_X(j) written] PV_X(j) -> commit p_free_X
//   softmax X: [S_X(j) ready] load S -> signal S free -> row max ->
//              exponentials of keys [0,64) -> [PV_X(j-1) done] rescale O if
//              needed, write P_X(j) keys [0,64) -> exponentials and P of keys
//              [64,128) -> signal
// K/V slots are loaded in the order the MMAs need them:
//   K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}.
// Stagger: QK_L(0) waits until the softmax of tile H has copied S_H(0) into
// registers, so the two tiles' softmax chains run a few hundred cycles apart
// instead of in lockstep (their exponentials, tensor-memory loads and P
// stores then contend less for the same units; measured 1.4-3.6 % faster at
// d = 128, no change at d = 64).
//
// Online softmax (M4.3 0x07-0x09; M4.6 0x09 conditional rescaling): each
// softmax thread keeps its row's retained reference r (raw score units) and
// denominator l in registers.  With lambda = scale*log2(e), a new tile with
// row maximum mx gives candidate c = max(r, mx); the reference moves only if
// (c - r)*lambda > 8, in which case l and the row of O are multiplied by
// gamma = 2^((r - c)*lambda).  P = 2^(lambda*s - lambda*r) <= 2^8 is rounded
// to the input dtype for the PV MMA while l accumulates the fp32 values.
// Epilogue: O = O / l,  LSE = (lambda*r + log2 l) * ln 2.
//
// Causal (M4.4 0x05.1A-D, bottom-right delta = Sk - Sq): key tiles wholly in
// the future are never loaded or multiplied; tiles crossing the diagonal or
// the key tail are masked element-wise to -inf before the row maximum.
#include <cuda_runtime.h>

#include "gbattn_internal.h"
#include "gbattn_ptx.cuh"

namespace gbattn {
namespace {

constexpr int kBM = 128;  // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kThreads = 384;
constexpr int kSoftmaxRegs = 224;
constexpr int kControlRegs = 56;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * 168, "register split");
constexpr int kMmaWarpH = 8;
constexpr int kLoadWarp = 9;
constexpr int kMmaWarpL = 10;
constexpr float kRescaleThreshold = 8.0f;  // log2 units (fp16/bf16 row of M4.6 0x09 table)

template <int D>
struct Cfg {
  // d = 64: P lives in tensor memory (the 128 columns S and O leave free) and
  // P.V reads it from there; d = 128: tensor memory is full, P is staged in
  // shared memory.
  static constexpr bool kPInTmem = (D == 64);
  static constexpr int kColBlocks = D / 64;           // 128-byte swizzle column blocks
  static constexpr int kTileBytes = kBM * D * 2;      // one 128 x D 16-bit tile
  static constexpr int kBlockBytes = kBM * 128;       // one 128-row x 128-byte block
  static constexpr int kPBytes = kPInTmem ? 0 : kBM * kBN * 2;  // one 128 x 128 16-bit P tile
  static constexpr int kStages = (D == 128) ? 3 : 8;  // K/V ring slots
  static constexpr int kQOff = 0;
  static constexpr int kPOff = 2 * kTileBytes;
  static constexpr int kRingOff = kPOff + 2 * kPBytes;
  static constexpr int kBarOff = kRingOff + kStages * kTileBytes;
  static constexpr int kSmemBytes = 1024 + kBarOff + 512;  // + alignment slack + barriers
};

struct Params {
  void* o;
  float* lse;
  int B, H, Hkv, Sq, Sk, g;
  int n_pairs;
  int head_group;
  int delta;
  float scale_log2;
  int causal;
  int* status;
  int wave;                       // CTAs resident at once (one per SM)
  unsigned long long* timeline;   // optional per-CTA records, or null
};

struct __align__(8) Barriers {
  uint64_t q_full;
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full[2];
  uint64_t p_free[2];     // P.V complete
  uint64_t o_full[2];
  uint64_t mma_done[2];
  uint64_t stagger;  // tile H has read its first S: tile L may start
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Number of key tiles query tile [q0, q0+128) visits (0 if the tile is empty
// or every row is fully masked): M4.4 0x05.1D n_block_max with the
// bottom-right offset.
__device__ __forceinline__ int tiles_for(int q0, int Sq, int Sk, int causal, int delta) {
  if (q0 >= Sq) return 0;
  const int nk = ceil_div(Sk, kBN);
  if (!causal) return nk;
  const int last_row = min(q0 + kBM - 1, Sq - 1);
  const int lim = last_row + delta;  // largest visible key of the tile
  if (lim < 0) return 0;
  return min(nk, lim / kBN + 1);
}

// Position of K_j / V_j in the load order K_0, K_1, V_0, K_2, V_1, ...,
// K_{n-1}, V_{n-2}, V_{n-1} (n key tiles).
__device__ __forceinline__ int item_of_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int item_of_v(int j, int n) { return j <= n - 2 ? 2 * j + 2 : 2 * n - 1; }

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q,
                       const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v,
                       const __grid_constant__ CUtensorMap tmap_o, const Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sP = smem + C::kPOff;
  uint8_t* sRing = smem + C::kRingOff;
  Barriers* bars = reinterpret_cast<Barriers*>(smem + C::kBarOff);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  unsigned long long t_start = 0;
  if (p.timeline != nullptr && threadIdx.x == 0) t_start = global_timer_ns();

  // ---- work unit.  CTAs are ordered in groups of p.head_group (batch, head)
  // pairs so that the K/V of the heads in flight stay resident in L2; inside
  // a group the heaviest query pairs (most causal key tiles) come first and
  // heads vary fastest (GQA heads sharing a KV head run side by side).
  const int BH = p.B * p.H;
  const int group = blockIdx.x / (p.head_group * p.n_pairs);
  const int heads_here = min(p.head_group, BH - group * p.head_group);
  const int r_in = blockIdx.x - group * p.head_group * p.n_pairs;
  const int bh = group * p.head_group + r_in % heads_here;
  const int pair = p.n_pairs - 1 - r_in / heads_here;
  const int b = bh / p.H;
  const int h = bh % p.H;
  const int kvh = h / p.g;
  // Per-tile first query row and key-tile count (scalars, not arrays: the
  // roles index them with a runtime tile number).
  const int q0_h = pair * 2 * kBM, q0_l = q0_h + kBM;
  const int nt_h = tiles_for(q0_h, p.Sq, p.Sk, CAUSAL ? 1 : 0, p.delta);
  const int nt_l = tiles_for(q0_l, p.Sq, p.Sk, CAUSAL ? 1 : 0, p.delta);
  const int n_max = max(nt_h, nt_l);

  // ---- K/V load items in the order K_0, K_1, V_0, K_2, V_1, ... (loader lane)
  const int n_items = 2 * n_max;
  auto issue_item = [&](int it, uint64_t policy) {
    const int st = it % C::kStages;
    bool is_v;
    int jt;
    if (it == 0) {
      is_v = false, jt = 0;
    } else if (it & 1) {
      if (it == n_items - 1) is_v = true, jt = n_max - 1;
      else is_v = false, jt = (it + 1) / 2;
    } else {
      is_v = true, jt = (it - 2) / 2;
    }
    mbar_arrive_expect_tx(&bars->kv_full[st], C::kTileBytes);
    for (int cb = 0; cb < C::kColBlocks; ++cb)
      tma_load_3d(sRing + st * C::kTileBytes + cb * C::kBlockBytes, is_v ? &tmap_v : &tmap_k, &bars->kv_full[st],
                  cb * 64, jt * kBN, b * p.Hkv + kvh, policy);
  };

  // ---- setup.  The loader lane initialises the load barriers itself and
  // requests Q and the first ring's worth of K/V (whose slots start free)
  // before the CTA-wide barrier, so those copies overlap the TMEM allocation
  // and the barrier.
  int pre_issued = 0;
  if (warp == kLoadWarp && lane == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 2);  // released by both MMA issuers
    }
    fence_mbar_init();
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
    prefetch_tensormap(&tmap_o);
    const uint64_t once = policy_evict_first();  // Q: read by this CTA only
    uint32_t q_bytes = 0;
    q_bytes += nt_h > 0 ? C::kTileBytes : 0;
    q_bytes += nt_l > 0 ? C::kTileBytes : 0;
    mbar_arrive_expect_tx(&bars->q_full, q_bytes);
    for (int x = 0; x < 2; ++x) {
      if ((x ? nt_l : nt_h) == 0) continue;
      for (int cb = 0; cb < C::kColBlocks; ++cb)
        tma_load_3d(sQ + x * C::kTileBytes + cb * C::kBlockBytes, &tmap_q, &bars->q_full, cb * 64,
                    x ? q0_l : q0_h, b * p.H + h, once);
    }
    const uint64_t keep = policy_evict_last();  // K/V: re-read by other CTAs
    pre_issued = min(C::kStages, n_items);
    for (int it = 0; it < pre_issued; ++it) issue_item(it, keep);
    // Q of the unit one wave ahead (the CTA that will most likely start on
    // an SM when the current wave drains) into L2, so that its first load
    // is not an HBM round trip.
    const int ahead = blockIdx.x + p.wave;
    if (ahead < static_cast<int>(gridDim.x)) {
      const int ga = ahead / (p.head_group * p.n_pairs);
      const int heads_a = min(p.head_group, BH - ga * p.head_group);
      const int ra = ahead - ga * p.head_group * p.n_pairs;
      const int bh_a = ga * p.head_group + ra % heads_a;
      const int pair_a = p.n_pairs - 1 - ra / heads_a;
      for (int x = 0; x < 2; ++x) {
        const int qa = (2 * pair_a + x) * kBM;
        if (qa >= p.Sq) continue;
        for (int cb = 0; cb < C::kColBlocks; ++cb) tma_prefetch_l2_3d(&tmap_q, cb * 64, qa, bh_a);
      }
    }
  }
  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars->s_full[x], 1);
      mbar_init(&bars->s_free[x], kBM);
      mbar_init(&bars->p_full[x], kBM);
      mbar_init(&bars->p_free[x], 1);
      mbar_init(&bars->o_full[x], 1);
      mbar_init(&bars->mma_done[x], 1);
    }
    mbar_init(&bars->stagger, kBM);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarpH) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp >= 8) {
    // ---- control warpgroup: TMA loader and MMA issuers
    regs_dec<kControlRegs>();
    if (warp == kLoadWarp) {
      // ================================================================ loader
      if (lane == 0) {
        const uint64_t keep = policy_evict_last();  // K/V: re-read by other CTAs
        int issued = pre_issued;
        for (int it = pre_issued; it < n_items; ++it) {
          const int st = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          if (!bounded_wait(&bars->kv_empty[st], ph ^ 1, abort_flag, p.status, kStatusTimeoutLoad))
            break;
          issue_item(it, keep);
          issued = it + 1;
        }
        // Drain: every copy this thread issued must have landed before exit.
        bounded_wait(&bars->q_full, 0, abort_flag, p.status, kStatusTimeoutDrain);
        for (int it = max(0, issued - C::kStages); it < issued; ++it) {
          const int st = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          int dummy = 0;
          // Ignore the abort flag here: wait for the copy itself (bounded).
          bounded_wait(&bars->kv_full[st], ph, reinterpret_cast<volatile int*>(&dummy), p.status,
                       kStatusTimeoutDrain);
        }
      }
      __syncwarp();
    } else if (warp == kMmaWarpH || warp == kMmaWarpL) {
      // ================================================================ MMA issuers
      // One issuing thread per query tile.  Both release every K/V slot (the
      // empty barriers count two arrivals); key tiles a query tile does not
      // visit (causal: H needs one fewer than L) are released once landed.
      if (lane == 0) {
        const int x = (warp == kMmaWarpH) ? 0 : 1;
        const int nt = x ? nt_l : nt_h;
        constexpr uint32_t kIdescQK = idesc_f16(BF16, false, false, kBM, kBN);
        constexpr uint32_t kIdescPV = idesc_f16(BF16, false, true, kBM, D);
        const uint32_t ring_addr = smem_u32(sRing);
        const uint32_t s_col = tmem + x * kBN;
        const uint32_t o_col = tmem + 2 * kBN + x * D;
        // Descriptors are built once; a K-step only adds (byte offset >> 4)
        // to the start-address field (every offset stays inside its tile).
        const uint64_t q_desc = smem_desc_sw128(smem_u32(sQ + x * C::kTileBytes), 16, 1024);
        const uint64_t p_desc = smem_desc_sw128(smem_u32(sP + x * C::kPBytes), 16, 1024);
        auto slot_of = [&](int item, uint32_t& parity) {
          parity = (item / C::kStages) & 1;
          return item % C::kStages;
        };
        auto issue_qk = [&](int st) {
          const uint64_t kd = smem_desc_sw128(ring_addr + st * C::kTileBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = ((kk / 4) * C::kBlockBytes + (kk % 4) * 32) >> 4;
            mma_f16_ss(s_col, q_desc + off, kd + off, kIdescQK, kk > 0 ? 1u : 0u);
          }
        };
        // P_X in tensor memory (d = 64): lane = query row, column c holds keys
        // (2c, 2c+1); a 16-key step of P.V reads 8 columns.
        const uint32_t p_tcol = tmem + 2 * kBN + 2 * D + x * (kBN / 2);
        // P.V over keys [64 half, 64 half + 64): P column block `half`
        auto issue_pv_half = [&](int st, int half, bool accumulate) {
          const uint64_t vd = smem_desc_sw128(ring_addr + st * C::kTileBytes, C::kBlockBytes, 1024);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = half * 4 + k4;
            const uint32_t acc = (accumulate || kk > 0) ? 1u : 0u;
            if constexpr (C::kPInTmem) {
              mma_f16_ts(o_col, p_tcol + kk * 8, vd + ((kk * 2048) >> 4), kIdescPV, acc);
            } else {
              const uint64_t poff = (half * C::kBlockBytes + k4 * 32) >> 4;
              mma_f16_ss(o_col, p_desc + poff, vd + ((kk * 2048) >> 4), kIdescPV, acc);
            }
          }
        };
        bool ok = nt == 0 || bounded_wait(&bars->q_full, 0, abort_flag, p.status, kStatusTimeoutMma);
        // Tile L's first QK waits until tile H has read S_H(0), so the two
        // tiles' softmax chains run staggered instead of in lockstep.
        if (ok && x == 1 && nt_h > 0 && nt_l > 0)
          ok = bounded_wait(&bars->stagger, 0, abort_flag, p.status, kStatusTimeoutMma);
        // S_X(0)
        if (ok && nt > 0) {
          uint32_t par;
          const int st = slot_of(item_of_k(0), par);
          ok = bounded_wait(&bars->kv_full[st], par, abort_flag, p.status, kStatusTimeoutMma);
          if (ok) {
            issue_qk(st);
            mma_commit(&bars->s_full[x]);
            mma_commit(&bars->kv_empty[st]);
          }
        }
        for (int j = 0; ok && j < nt; ++j) {
          // QK_X(j+1) once the softmax threads hold S_X(j) in registers
          if (j + 1 < nt) {
            uint32_t par;
            const int st = slot_of(item_of_k(j + 1), par);
            if (!(ok = bounded_wait(&bars->kv_full[st], par, abort_flag, p.status, kStatusTimeoutMma)))
              break;
            if (!(ok = bounded_wait(&bars->s_free[x], j & 1, abort_flag, p.status, kStatusTimeoutMma)))
              break;
            tc_fence_after();
            issue_qk(st);
            mma_commit(&bars->s_full[x]);
            mma_commit(&bars->kv_empty[st]);
          }
          // PV_X(j) once P_X(j) is in shared memory (and O_X corrected)
          {
            uint32_t par;
            const int st = slot_of(item_of_v(j, n_max), par);
            if (!(ok = bounded_wait(&bars->kv_full[st], par, abort_flag, p.status, kStatusTimeoutMma)))
              break;
            if (!(ok = bounded_wait(&bars->p_full[x], j & 1, abort_flag, p.status, kStatusTimeoutMma)))
              break;
            tc_fence_after();
            issue_pv_half(st, 0, j > 0);
            issue_pv_half(st, 1, true);
            mma_commit(&bars->p_free[x]);
            if (j == nt - 1) mma_commit(&bars->o_full[x]);
            mma_commit(&bars->kv_empty[st]);
          }
        }
        // Release the K/V slots of key tiles this query tile does not visit.
        for (int j = nt; ok && j < n_max; ++j) {
          for (int kv = 0; kv < 2; ++kv) {
            uint32_t par;
            const int st = slot_of(kv ? item_of_v(j, n_max) : item_of_k(j), par);
            if (!(ok = bounded_wait(&bars->kv_full[st], par, abort_flag, p.status, kStatusTimeoutMma)))
              break;
            mbar_arrive(&bars->kv_empty[st]);
          }
        }
        // Every MMA this thread issued must complete before TMEM is released.
        mma_commit(&bars->mma_done[x]);
        int dummy = 0;
        bounded_wait(&bars->mma_done[x], 0, reinterpret_cast<volatile int*>(&dummy), p.status,
                     kStatusTimeoutDrain);
      }
      __syncwarp();
    }
  } else {
    // ---- softmax warpgroups
    regs_inc<kSoftmaxRegs>();
    // ================================================================ softmax
    const int x = warp / 4;     // 0 = tile H, 1 = tile L
    const int wq = warp % 4;    // TMEM lane quarter owned by this warp
    const int row = wq * 32 + lane;
    const int q0x = x ? q0_l : q0_h;
    const int q_row = q0x + row;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_tmem = tmem + lane_off + x * kBN;
    const uint32_t o_tmem = tmem + lane_off + 2 * kBN + x * D;
    // This row of P_X in shared memory: two 64-key column blocks of 128-byte
    // rows; 16-byte chunk c of the row sits at chunk c ^ (row % 8).
    uint8_t* p_row = sP + x * C::kPBytes + row * 128;
    const uint32_t p_tmem = tmem + lane_off + 2 * kBN + 2 * D + x * (kBN / 2);  // d = 64
    const float lam = p.scale_log2;
    float r = -INFINITY;  // retained reference, raw score units
    float l = 0.f;
    bool ok = true;
    const int nt = x ? nt_l : nt_h;

    for (int j = 0; j < nt; ++j) {
      ok = bounded_wait(&bars->s_full[x], j & 1, abort_flag, p.status, kStatusTimeoutSoftmax);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int k0 = j * kBN;
      const bool tail = k0 + kBN > p.Sk;
      const bool diag = CAUSAL && (k0 + kBN - 1 > q0x + p.delta);
      // ---- S row -> registers (four loads in flight, one wait), then S_X is free
      uint32_t u[kBN];
      float mq[kBN / 32];
      if (tail || diag) {
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
      mbar_arrive(&bars->s_free[x]);
      if (x == 0 && j == 0 && nt_l > 0) mbar_arrive(&bars->stagger);
      float* s = reinterpret_cast<float*>(u);
      float mx;
      if (tail || diag) {
        const int lim = CAUSAL ? min(p.Sk - 1, q_row + p.delta) : p.Sk - 1;  // last visible key
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (k0 + c > lim) s[c] = -INFINITY;
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
        // the loads returned each 32-column block's maximum
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
      // ---- P = 2^(lambda*s - lambda*r), row sum, pack to 16 bits, and store
      // the row of P_X(j) as the A operand of P.V (d = 128: shared memory,
      // swizzled K-major; d = 64: this row's tensor-memory lane), one 64-key
      // column block at a time.  Before block 0 is stored, PV_X(j-1) must be
      // complete: it has then read all of P_X(j-1) and O_X is stable, so the
      // correction happens there.  (Releasing P in two halves, a commit after
      // the P.V steps over keys [0,64), adds a commit to the issuer and a wait
      // to this chain: measured 1.8-1.9 % slower at d = 128 causal and GQA,
      // 0.7 % non-causal, 8.6 % at d = 64.)
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
        if (j > 0 && blk == 0) {
          ok = bounded_wait(&bars->p_free[x], (j - 1) & 1, abort_flag, p.status, kStatusTimeoutSoftmax);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();  // P.V(j-1) is complete: P may be overwritten, O_X is stable
          // correction: O_row *= gamma (warp-uniform path; gamma = 1 rows unchanged)
          if (__any_sync(0xffffffffu, gamma != 1.f)) {
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
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
        }
        if constexpr (C::kPInTmem) {
          tmem_st32(p_tmem + blk * 32, pk);
        } else {
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8)
            *reinterpret_cast<uint4*>(p_row + blk * C::kBlockBytes + ((c8 ^ (row & 7)) << 4)) =
                make_uint4(pk[c8 * 4], pk[c8 * 4 + 1], pk[c8 * 4 + 2], pk[c8 * 4 + 3]);
        }
      }
      if (!ok) break;
      const float2 s01 = fadd2(fadd2(sum4[0], sum4[1]), fadd2(sum4[2], sum4[3]));
      l += s01.x + s01.y;
      if constexpr (C::kPInTmem) {
        tmem_wait_st();            // P (tcgen05.st) complete before the arrive
      } else {
        fence_proxy_async_smem();  // P stores -> visible to the tensor core (async proxy)
      }
      tc_fence_before();           // P / O correction (tcgen05.st) ordered before the arrive
      mbar_arrive(&bars->p_full[x]);
    }

    // ---- epilogue: O = O / l, LSE
    if (q0x < p.Sq) {
      bool have_o = false;
      if (ok && nt > 0) {
        have_o = bounded_wait(&bars->o_full[x], 0, abort_flag, p.status, kStatusTimeoutSoftmax);
        have_o = __all_sync(0xffffffffu, have_o);
        tc_fence_after();
      }
      const bool row_ok = q_row < p.Sq;
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      // O_X is staged in Q_X (dead since QK_X of the last key tile completed)
      // in the Q layout -- 64-element column blocks of 128-byte rows, 16-byte
      // chunk c at chunk c ^ (row % 8) -- and written by one TMA store per
      // column block (rows past Sq are not written).  Each thread storing its
      // own row to global memory instead costs one cache line per lane and
      // store instruction: ~4,000 line writes per CTA, ~1.8 us (traced).
      uint8_t* o_row = sQ + x * C::kTileBytes + row * 128;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        if (have_o) {
          tmem_ld32(o_tmem + c * 32, u);
          tmem_wait_ld();
          reg_fence32(u);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2<BF16>(__uint_as_float(u[2 * i]) * inv, __uint_as_float(u[2 * i + 1]) * inv);
        uint8_t* blk = o_row + (c / 2) * C::kBlockBytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int ch = (c % 2) * 4 + k;
          *reinterpret_cast<uint4*>(blk + ((ch ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
      }
      fence_proxy_async_smem();    // O stores -> visible to the TMA engine
      named_bar_sync(1 + x, kBM);  // the four warps of the tile have written O_X
      if (wq == 0 && lane == 0) {
        for (int cb = 0; cb < C::kColBlocks; ++cb)
          tma_store_3d(&tmap_o, sQ + x * C::kTileBytes + cb * C::kBlockBytes, cb * 64, q0x, b * p.H + h);
        bulk_commit_group();
        bulk_wait_group_read0();  // shared memory read before the CTA may exit
      }
      if (row_ok && p.lse != nullptr) {
        const float lse = (l > 0.f) ? (r * lam + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        p.lse[(static_cast<size_t>(b) * p.H + h) * p.Sq + q_row] = lse;
      }
    }
  }

  // ---- teardown: all TMEM traffic done before the allocator warp frees it
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (p.timeline != nullptr && threadIdx.x == 0) {
    // Timeline record of this CTA: start and end (%globaltimer ns), SM, unit.
    unsigned long long* rec = p.timeline + 4 * static_cast<size_t>(blockIdx.x);
    rec[0] = t_start;
    rec[1] = global_timer_ns();
    rec[2] = sm_id();
    rec[3] = static_cast<unsigned long long>(bh) << 32 | static_cast<unsigned>(pair);
  }
  if (warp == kMmaWarpH) tmem_dealloc(tmem, 512);
}

template <int D, bool BF16, bool CAUSAL>
int launch_t(const PrefillArgs& a) {
  using C = Cfg<D>;
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap_3d(&tq, a.q, BF16, D, a.Sq, static_cast<long long>(a.B) * a.H, kBM) ||
      !make_tmap_3d(&to, a.o, BF16, D, a.Sq, static_cast<long long>(a.B) * a.H, kBM) ||
      !make_tmap_3d(&tk, a.k, BF16, D, a.Sk, static_cast<long long>(a.B) * a.Hkv, kBN) ||
      !make_tmap_3d(&tv, a.v, BF16, D, a.Sk, static_cast<long long>(a.B) * a.Hkv, kBN))
    return -1;
  auto kern = prefill_fwd_kernel<D, BF16, CAUSAL>;
  static std::atomic<unsigned long long> attr_done{0};  // per instantiation
  if (!set_smem_limit_once(kern, C::kSmemBytes, attr_done)) return -1;
  Params p{};
  p.o = a.o;
  p.lse = a.lse;
  p.B = a.B;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Sk = a.Sk;
  p.g = a.H / a.Hkv;
  p.n_pairs = (a.Sq + 2 * kBM - 1) / (2 * kBM);
  {
    // Heads per scheduling group: about 48 MB of K/V in flight (L2 is 129 MB),
    // whole KV-head groups, groups of equal size (balanced_head_group).
    const long long kv_head_bytes = 4LL * a.Sk * D;  // K and V, 16-bit
    long long kv_heads = (48LL << 20) / (kv_head_bytes > 0 ? kv_head_bytes : 1);
    if (kv_heads < 1) kv_heads = 1;
    p.head_group = balanced_head_group(kv_heads * p.g, static_cast<long long>(a.B) * a.H, p.g);
  }
  p.delta = a.Sk - a.Sq;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.causal = CAUSAL ? 1 : 0;
  p.status = a.status;
  p.wave = a.num_sms;
  const long long grid = static_cast<long long>(a.B) * a.H * p.n_pairs;
  if (grid > 0x7FFFFFFFLL) return -1;
  p.timeline = (a.timeline != nullptr && a.timeline_capacity >= grid) ? a.timeline : nullptr;
  kern<<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, a.stream>>>(tq, tk, tv, to, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_prefill(const PrefillArgs& a) {
  if (a.d == 128) {
    if (a.bf16) return a.causal ? launch_t<128, true, true>(a) : launch_t<128, true, false>(a);
    return a.causal ? launch_t<128, false, true>(a) : launch_t<128, false, false>(a);
  }
  if (a.bf16) return a.causal ? launch_t<64, true, true>(a) : launch_t<64, true, false>(a);
  return a.causal ? launch_t<64, false, true>(a) : launch_t<64, false, false>(a);
}

}  // namespace gbattn
