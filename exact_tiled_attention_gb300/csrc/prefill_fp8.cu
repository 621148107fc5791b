// prefill_fp8.cu -- exact attention forward with E4M3 (FP8) Q, K, V on
// sm_103a: the FP8 path of M4.6 "FlashAttention-3/4 Hardware Pipelines"
// 0x06, on the same two-query-tile, TMA + tcgen05 + TMEM structure as the
// 16-bit forward (prefill_fwd.cu), head dimension 128.
//
// Arithmetic (0x06 "Derive Where Every Scale Must Enter"): with per-(batch,
// KV head) descales dQ, dK, dV (the pinned public API's [batch, kv_head]
// granularity; absent descales are 1),
//     S  = (scale dQ dK) Q8 K8^T          fp32 in TMEM (kind::f8f6f4 MMA)
//     u  = 2^omega exp(S - r)             fp32, omega = 4 (log2 units)
//     P8 = E4M3(u)                        the A operand of the P.V product
//     O  = dV (sum_j P8_j V8_j) / (sum_j u_j)   fp32 accumulation, bf16 out
//     LSE = r + log(sum_j u_j) - omega ln 2
// The probability offset 2^omega and the conditional-rescale threshold
// tau = 4 (log2 units) bound every u by 2^(tau + omega) = 256 <= 448, the
// E4M3 maximum (M4.6 0x09 "Threshold And Probability Offset Form One Range
// Contract", FP8 E4M3FN row); the offset cancels between numerator and
// denominator.
//
// Layout (0x06 "FP8 WGMMA Turns V Layout Into A Producer Job"): both 8-bit
// operands of each product are read K-major.  Q and K are contiguous in d,
// the reduction axis of Q K^T; for P V the reduction axis is the key axis, so
// a first kernel writes V^T [B, Hkv, d, Sk_pad] into the caller's workspace
// (the "standalone global transpose" design of that section's table).
//
// Tiles are 128 rows x 128 bytes (one 128-byte swizzle block): Q_H, Q_L,
// two P buffers per query tile and an 8-slot ring of K / V^T tiles, 16 KiB
// each.  One MMA instruction is 128 x 128 x 32.
//
// As in the 16-bit forward, tile L's first QK waits until tile H's softmax
// has copied S_H(0) into registers (the two softmax chains run staggered).
// P(j) goes to buffer j mod 2, last read by P.V(j-2); the issuer issues
// QK(j) after P.V(j-2), and a commit covers every earlier MMA of its
// thread, so S(j) ready implies that buffer free and the softmax has no P
// wait of its own (only a correction of O waits for P.V(j-1)).  Measured on
// the causal [4,16,8192,128] workload: 0.677 ms with P released in two
// halves and a lockstep start, 0.619 ms with one release per key tile and
// the stagger, 0.604 ms with the second buffer.
#include <cuda_runtime.h>

#include "gbattn_internal.h"
#include "gbattn_ptx.cuh"

namespace gbattn {
namespace {

constexpr int kD = 128;
constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per tile
constexpr int kThreads = 384;
constexpr int kSoftmaxRegs = 224;
constexpr int kControlRegs = 56;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * 168, "register split");
constexpr int kMmaWarpH = 8;
constexpr int kLoadWarp = 9;
constexpr int kMmaWarpL = 10;
constexpr float kTau = 4.0f;    // conditional-rescale threshold, log2 units
constexpr float kOmega = 4.0f;  // probability offset, log2 units
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kTile = kBM * 128;  // 16 KiB
constexpr int kStages = 8;        // K / V^T ring slots
constexpr int kQOff = 0;
constexpr int kPOff = 2 * kTile;
constexpr int kRingOff = 6 * kTile;  // Q_H, Q_L, P_H[2], P_L[2]
constexpr int kBarOff = kRingOff + kStages * kTile;
constexpr int kSmemBytes = 1024 + kBarOff + 512;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// Instruction descriptor, kind::f8f6f4: D fp32 (bits 4-5 = 1), A and B E4M3
// (format code 0 in bits 7-9 and 10-12), both K-major, N >> 3 at bit 17,
// M >> 4 at bit 24.
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(kBN >> 3) << 17) |
                            (static_cast<uint32_t>(kBM >> 4) << 24);
static_assert(kBN == kD, "QK^T and P.V share one instruction shape");

struct Fp8Params {
  void* o;
  float* lse;
  const float* dq;
  const float* dk;
  const float* dv;
  int B, H, Hkv, Sq, Sk, g;
  int n_pairs, head_group, delta;
  float scale;
  int* status;
  int wave;                       // CTAs resident at once (one per SM)
  unsigned long long* timeline;   // optional per-CTA records, or null
};

struct __align__(8) Bars {
  uint64_t q_full;
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
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
static_assert(sizeof(Bars) <= 512, "barrier block");

__device__ __forceinline__ int tiles_for(int q0, int Sq, int Sk, bool causal, int delta) {
  if (q0 >= Sq) return 0;
  const int nk = (Sk + kBN - 1) / kBN;
  if (!causal) return nk;
  const int lim = min(q0 + kBM - 1, Sq - 1) + delta;  // largest visible key of the tile
  if (lim < 0) return 0;
  return min(nk, lim / kBN + 1);
}

// Load order K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}.
__device__ __forceinline__ int item_of_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int item_of_v(int j, int n) { return j <= n - 2 ? 2 * j + 2 : 2 * n - 1; }

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_fp8_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_vt, const __grid_constant__ CUtensorMap tmap_o,
                       const Fp8Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + kQOff;
  uint8_t* sP = smem + kPOff;
  uint8_t* sRing = smem + kRingOff;
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  unsigned long long t_start = 0;
  if (p.timeline != nullptr && threadIdx.x == 0) t_start = global_timer_ns();

  // ---- work unit (same order as the 16-bit forward): groups of heads whose
  // K/V stay in L2, heaviest causal query pairs first, heads fastest.
  const int BH = p.B * p.H;
  const int group = blockIdx.x / (p.head_group * p.n_pairs);
  const int heads_here = min(p.head_group, BH - group * p.head_group);
  const int r_in = blockIdx.x - group * p.head_group * p.n_pairs;
  const int bh = group * p.head_group + r_in % heads_here;
  const int pair = p.n_pairs - 1 - r_in / heads_here;
  const int b = bh / p.H;
  const int h = bh % p.H;
  const int kvh = h / p.g;
  const int bkv = b * p.Hkv + kvh;
  const int q0_h = pair * 2 * kBM, q0_l = q0_h + kBM;
  const int nt_h = tiles_for(q0_h, p.Sq, p.Sk, CAUSAL, p.delta);
  const int nt_l = tiles_for(q0_l, p.Sq, p.Sk, CAUSAL, p.delta);
  const int n_max = max(nt_h, nt_l);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 2);  // released by both MMA issuers
    }
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
  if (warp == kLoadWarp && lane == 0) {
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_vt);
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
    regs_dec<kControlRegs>();
    if (warp == kLoadWarp) {
      // ================================================================ loader
      if (lane == 0) {
        const uint64_t keep = policy_evict_last();   // K/V^T: re-read by other CTAs
        const uint64_t once = policy_evict_first();  // Q: read by this CTA only
        mbar_arrive_expect_tx(&bars->q_full, (nt_h > 0 ? kTile : 0) + (nt_l > 0 ? kTile : 0));
        if (nt_h > 0) tma_load_3d(sQ, &tmap_q, &bars->q_full, 0, q0_h, b * p.H + h, once);
        if (nt_l > 0) tma_load_3d(sQ + kTile, &tmap_q, &bars->q_full, 0, q0_l, b * p.H + h, once);
        {  // Q of the unit one wave ahead into L2 (as in the 16-bit forward)
          const int ahead = blockIdx.x + p.wave;
          if (ahead < static_cast<int>(gridDim.x)) {
            const int ga = ahead / (p.head_group * p.n_pairs);
            const int heads_a = min(p.head_group, BH - ga * p.head_group);
            const int ra = ahead - ga * p.head_group * p.n_pairs;
            const int bh_a = ga * p.head_group + ra % heads_a;
            const int pair_a = p.n_pairs - 1 - ra / heads_a;
            for (int x = 0; x < 2; ++x) {
              const int qa = (2 * pair_a + x) * kBM;
              if (qa < p.Sq) tma_prefetch_l2_3d(&tmap_q, 0, qa, bh_a);
            }
          }
        }
        const int n_items = 2 * n_max;
        int issued = 0;
        for (int it = 0; it < n_items; ++it) {
          const int st = it % kStages;
          if (!bounded_wait(&bars->kv_empty[st], ((it / kStages) & 1) ^ 1, abort_flag, p.status,
                            kStatusTimeoutLoad))
            break;
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
          mbar_arrive_expect_tx(&bars->kv_full[st], kTile);
          if (is_v)  // V^T rows are d, its columns keys: the tile starts at key jt * 128
            tma_load_3d(sRing + st * kTile, &tmap_vt, &bars->kv_full[st], jt * kBN, 0, bkv, keep);
          else
            tma_load_3d(sRing + st * kTile, &tmap_k, &bars->kv_full[st], 0, jt * kBN, bkv, keep);
          issued = it + 1;
        }
        bounded_wait(&bars->q_full, 0, abort_flag, p.status, kStatusTimeoutDrain);
        int dummy = 0;
        for (int it = max(0, issued - kStages); it < issued; ++it)
          bounded_wait(&bars->kv_full[it % kStages], (it / kStages) & 1, reinterpret_cast<volatile int*>(&dummy),
                       p.status, kStatusTimeoutDrain);
      }
      __syncwarp();
    } else if (warp == kMmaWarpH || warp == kMmaWarpL) {
      // ================================================================ MMA issuers
      if (lane == 0) {
        const int x = (warp == kMmaWarpH) ? 0 : 1;
        const int nt = x ? nt_l : nt_h;
        const uint32_t ring_addr = smem_u32(sRing);
        const uint32_t s_col = tmem + x * kBN;
        const uint32_t o_col = tmem + 2 * kBN + x * kD;
        const uint64_t q_desc = smem_desc_sw128(smem_u32(sQ + x * kTile), 16, 1024);
        const uint64_t p_desc0 = smem_desc_sw128(smem_u32(sP + 2 * x * kTile), 16, 1024);
        auto slot_of = [&](int item, uint32_t& parity) {
          parity = (item / kStages) & 1;
          return item % kStages;
        };
        // a K-step is 32 one-byte elements = 32 bytes inside the 128-byte row
        auto issue_qk = [&](int st) {
          const uint64_t kd = smem_desc_sw128(ring_addr + st * kTile, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kD / 32; ++kk) mma_f8_ss(s_col, q_desc + kk * 2, kd + kk * 2, kIdesc, kk > 0 ? 1u : 0u);
        };
        auto issue_pv_steps = [&](int st, int kk0, int kk1, bool accumulate, int pbuf) {
          const uint64_t vd = smem_desc_sw128(ring_addr + st * kTile, 16, 1024);
          const uint64_t p_desc = p_desc0 + ((pbuf * kTile) >> 4);
#pragma unroll
          for (int kk = kk0; kk < kk1; ++kk)
            mma_f8_ss(o_col, p_desc + kk * 2, vd + kk * 2, kIdesc, (accumulate || kk > 0) ? 1u : 0u);
        };
        bool ok = nt == 0 || bounded_wait(&bars->q_full, 0, abort_flag, p.status, kStatusTimeoutMma);
        // Tile L's first QK waits until tile H has read S_H(0) (staggered softmax chains).
        if (ok && x == 1 && nt_h > 0 && nt_l > 0)
          ok = bounded_wait(&bars->stagger, 0, abort_flag, p.status, kStatusTimeoutMma);
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
          if (j + 1 < nt) {
            uint32_t par;
            const int st = slot_of(item_of_k(j + 1), par);
            if (!(ok = bounded_wait(&bars->kv_full[st], par, abort_flag, p.status, kStatusTimeoutMma))) break;
            if (!(ok = bounded_wait(&bars->s_free[x], j & 1, abort_flag, p.status, kStatusTimeoutMma))) break;
            tc_fence_after();
            issue_qk(st);
            mma_commit(&bars->s_full[x]);
            mma_commit(&bars->kv_empty[st]);
          }
          {
            uint32_t par;
            const int st = slot_of(item_of_v(j, n_max), par);
            if (!(ok = bounded_wait(&bars->kv_full[st], par, abort_flag, p.status, kStatusTimeoutMma))) break;
            if (!(ok = bounded_wait(&bars->p_full[x], j & 1, abort_flag, p.status, kStatusTimeoutMma))) break;
            tc_fence_after();
            issue_pv_steps(st, 0, 4, j > 0, j & 1);
            mma_commit(&bars->p_free[x]);
            if (j == nt - 1) mma_commit(&bars->o_full[x]);
            mma_commit(&bars->kv_empty[st]);
          }
        }
        // Release the slots of key tiles this query tile does not visit.
        for (int j = nt; ok && j < n_max; ++j) {
          for (int kv = 0; kv < 2; ++kv) {
            uint32_t par;
            const int st = slot_of(kv ? item_of_v(j, n_max) : item_of_k(j), par);
            if (!(ok = bounded_wait(&bars->kv_full[st], par, abort_flag, p.status, kStatusTimeoutMma))) break;
            mbar_arrive(&bars->kv_empty[st]);
          }
        }
        mma_commit(&bars->mma_done[x]);
        int dummy = 0;
        bounded_wait(&bars->mma_done[x], 0, reinterpret_cast<volatile int*>(&dummy), p.status, kStatusTimeoutDrain);
      }
      __syncwarp();
    }
  } else {
    // ================================================================ softmax
    regs_inc<kSoftmaxRegs>();
    const int x = warp / 4;
    const int wq = warp % 4;
    const int row = wq * 32 + lane;
    const int q0x = x ? q0_l : q0_h;
    const int q_row = q0x + row;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_tmem = tmem + lane_off + x * kBN;
    const uint32_t o_tmem = tmem + lane_off + 2 * kBN + x * kD;
    uint8_t* p_row0 = sP + 2 * x * kTile + row * 128;  // buffer b at + b * kTile
    const float dqk = (p.dq ? p.dq[bkv] : 1.f) * (p.dk ? p.dk[bkv] : 1.f);
    const float dvs = p.dv ? p.dv[bkv] : 1.f;
    const float lam = p.scale * dqk * kLog2e;  // log2 units per raw Q8.K8 score
    float r = -INFINITY;
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
      const bool masked = (k0 + kBN > p.Sk) || (CAUSAL && (k0 + kBN - 1 > q0x + p.delta));
      // S row -> registers; an unmasked tile's loads also return each
      // 32-column block's maximum (tcgen05.ld.red)
      uint32_t u[kBN];
      float mq[kBN / 32];
      if (masked) {
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) tmem_ld32(s_tmem + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&u[c * 32]));
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
      if (masked) {
        const int lim = CAUSAL ? min(p.Sk - 1, q_row + p.delta) : p.Sk - 1;  // last visible key
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (k0 + c > lim) s[c] = -INFINITY;
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
        if ((cand - r) * lam > kTau) {
          gamma = ex2_approx((r - cand) * lam);
          r = cand;
        }
      }
      l *= gamma;
      // u = 2^(lambda s - lambda r + omega) <= 2^(tau + omega) = 256, then E4M3
      const float rs = (r == -INFINITY) ? 0.f : r * lam;
      const float2 lam2 = make_float2(lam, lam);
      const float2 nrs2 = make_float2(kOmega - rs, kOmega - rs);
      float2 sum4[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[16];  // 64 keys, four E4M3 codes per word
#pragma unroll
        for (int w = 0; w < 16; ++w) {
          const int c = half * 64 + w * 4;
          const float2 a = ffma2(make_float2(s[c], s[c + 1]), lam2, nrs2);
          const float2 e = ffma2(make_float2(s[c + 2], s[c + 3]), lam2, nrs2);
          // the build option GBATTN_EX2_EMU_EVERY sends every E-th pair to the
          // FMA-pipe exp2 (ex2_pair), as in the 16-bit kernels
          const float2 ta = ex2_pair(a, half * 32 + w * 2);
          const float2 te = ex2_pair(e, half * 32 + w * 2 + 1);
          sum4[0] = fadd2(sum4[0], ta);
          sum4[1] = fadd2(sum4[1], te);
          pk[w] = pack4_e4m3(ta.x, ta.y, te.x, te.y);
        }
        // P buffer j & 1 was last read by P.V(j-2), complete since s_full(j):
        // the issuer issues QK(j) after P.V(j-2).  Only a correction of O
        // waits for P.V(j-1).
        if (j > 0 && half == 0 && __any_sync(0xffffffffu, gamma != 1.f)) {
          ok = bounded_wait(&bars->p_free[x], (j - 1) & 1, abort_flag, p.status, kStatusTimeoutSoftmax);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          {  // correction O_row *= gamma
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
        }
        // 16-byte chunk ch (16 keys) of the 128-byte row at chunk ch ^ (row % 8)
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const int ch = half * 4 + c4;
          *reinterpret_cast<uint4*>(p_row0 + (j & 1) * kTile + ((ch ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
        }
      }
      if (!ok) break;
      const float2 s01 = fadd2(sum4[0], sum4[1]);
      l += s01.x + s01.y;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full[x]);
    }

    // ---- epilogue: O = dV O / l (the 2^omega of u cancels), LSE
    if (q0x < p.Sq) {
      bool have_o = false;
      if (ok && nt > 0) {
        have_o = bounded_wait(&bars->o_full[x], 0, abort_flag, p.status, kStatusTimeoutSoftmax);
        have_o = __all_sync(0xffffffffu, have_o);
        tc_fence_after();
      }
      const bool row_ok = q_row < p.Sq;
      const float mul = (l > 0.f) ? dvs / l : 0.f;
      // O_X (bf16, two 64-column blocks of 16 KiB) is staged in Q_X and P_X
      // (dead once the last P.V has completed), 128-byte rows with 16-byte
      // chunk c at chunk c ^ (row % 8), and written by two TMA stores (rows
      // past Sq are not written).
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
          pk[i] = pack2<true>(__uint_as_float(w[2 * i]) * mul, __uint_as_float(w[2 * i + 1]) * mul);
        uint8_t* blk = ((c / 2) ? sP + 2 * x * kTile : sQ + x * kTile) + row * 128;
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
        tma_store_3d(&tmap_o, sQ + x * kTile, 0, q0x, b * p.H + h);
        tma_store_3d(&tmap_o, sP + 2 * x * kTile, 64, q0x, b * p.H + h);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
      if (row_ok && p.lse != nullptr) {
        const float lse = (l > 0.f) ? (r * lam + __log2f(l) - kOmega) * 0.69314718055994531f : -INFINITY;
        p.lse[(static_cast<size_t>(b) * p.H + h) * p.Sq + q_row] = lse;
      }
    }
  }

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

// V [B*Hkv, Sk, 128] (bytes) -> V^T [B*Hkv, 128, Sk_pad]; keys in [Sk, Sk_pad)
// are written as zero.  One CTA per 64 keys of one (batch, KV head).
__global__ void __launch_bounds__(256) v_transpose_kernel(const uint8_t* __restrict__ v, uint8_t* __restrict__ vt,
                                                          int Sk, int Sk_pad) {
  __shared__ uint32_t tile[64][33];  // 64 key rows of 128 bytes (+4 bytes of padding)
  const int k0 = blockIdx.x * 64;
  const long long bkv = blockIdx.y;
  for (int i = threadIdx.x; i < 64 * 8; i += blockDim.x) {
    const int key = i / 8, c = i % 8;  // 16-byte chunk c of the key row
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (k0 + key < Sk) val = reinterpret_cast<const uint4*>(v + (bkv * Sk + k0 + key) * kD)[c];
    tile[key][4 * c] = val.x;
    tile[key][4 * c + 1] = val.y;
    tile[key][4 * c + 2] = val.z;
    tile[key][4 * c + 3] = val.w;
  }
  __syncthreads();
  const uint8_t* tb = reinterpret_cast<const uint8_t*>(&tile[0][0]);
  constexpr int kRow = 33 * 4;  // bytes per tile row
  for (int i = threadIdx.x; i < kD * 4; i += blockDim.x) {
    const int dd = i / 4, c = i % 4;  // output row dd, keys [16 c, 16 c + 16)
    uint32_t w[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      uint32_t word = 0;
#pragma unroll
      for (int bi = 0; bi < 4; ++bi) word |= static_cast<uint32_t>(tb[(16 * c + 4 * m + bi) * kRow + dd]) << (8 * bi);
      w[m] = word;
    }
    *reinterpret_cast<uint4*>(vt + (bkv * kD + dd) * Sk_pad + k0 + 16 * c) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <bool CAUSAL>
int launch_fp8_t(const PrefillFp8Args& a) {
  const int Sk_pad = (a.Sk + kBN - 1) / kBN * kBN;
  const long long BHkv = static_cast<long long>(a.B) * a.Hkv;
  if (BHkv > 65535) return -1;
  v_transpose_kernel<<<dim3(Sk_pad / 64, static_cast<unsigned>(BHkv)), 256, 0, a.stream>>>(
      static_cast<const uint8_t*>(a.v), static_cast<uint8_t*>(a.vt), a.Sk, Sk_pad);
  CUtensorMap tq, tk, tvt, to;
  if (!make_tmap_3d_u8(&tq, a.q, kD, a.Sq, static_cast<long long>(a.B) * a.H, kBM) ||
      !make_tmap_3d_u8(&tk, a.k, kD, a.Sk, BHkv, kBN) ||
      !make_tmap_3d_u8(&tvt, a.vt, Sk_pad, kD, BHkv, kD) ||
      !make_tmap_3d(&to, a.o, true, kD, a.Sq, static_cast<long long>(a.B) * a.H, kBM))
    return -1;
  auto kern = prefill_fp8_kernel<CAUSAL>;
  static std::atomic<unsigned long long> attr_done{0};  // per instantiation
  if (!set_smem_limit_once(kern, kSmemBytes, attr_done)) return -1;
  Fp8Params p{};
  p.o = a.o;
  p.lse = a.lse;
  p.dq = a.q_descale;
  p.dk = a.k_descale;
  p.dv = a.v_descale;
  p.B = a.B;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Sk = a.Sk;
  p.g = a.H / a.Hkv;
  p.n_pairs = (a.Sq + 2 * kBM - 1) / (2 * kBM);
  {
    // heads per scheduling group: about 48 MB of K and V^T (8-bit) in flight
    const long long kv_head_bytes = 2LL * a.Sk * kD;
    long long kv_heads = (48LL << 20) / (kv_head_bytes > 0 ? kv_head_bytes : 1);
    if (kv_heads < 1) kv_heads = 1;
    p.head_group = balanced_head_group(kv_heads * p.g, static_cast<long long>(a.B) * a.H, p.g);
  }
  p.delta = a.Sk - a.Sq;
  p.scale = a.scale;
  p.status = a.status;
  p.wave = a.num_sms;
  const long long grid = static_cast<long long>(a.B) * a.H * p.n_pairs;
  if (grid > 0x7FFFFFFFLL) return -1;
  p.timeline = (a.timeline != nullptr && a.timeline_capacity >= grid) ? a.timeline : nullptr;
  kern<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, a.stream>>>(tq, tk, tvt, to, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_prefill_fp8(const PrefillFp8Args& a) {
  if (a.d != kD) return -1;
  return a.causal ? launch_fp8_t<true>(a) : launch_fp8_t<false>(a);
}

}  // namespace gbattn
