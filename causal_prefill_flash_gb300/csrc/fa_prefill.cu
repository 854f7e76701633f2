// fa_prefill.cu -- causal prefill flash attention for GB300 (sm_103a).
//
//   O = softmax(scale * Q K^T + causal mask) V,  16-bit Q/K/V/O, f32 accumulate.
//
// The pages' kernel walks the KV tiles of one query tile keeping the running
// row max m and row sum l of the online softmax (minfer "53 · r50 — FA_TKV
// 32->16 occupancy experiment", section 2: stage K/V, S = Q K^T, mask, max,
// exp, sum, rescale O, O += P V).  It does that with wmma fragments and
// cp.async on another GPU; here the same steps are re-planned for Blackwell.
//
// One CTA owns TWO 128-row query tiles (A and B) that read the same K/V:
// two query heads of one GQA group at the same rows, or -- when a group has an
// odd number of query heads -- two consecutive row tiles of one head.  Both
// tiles share every K/V tile the CTA loads, halving K/V traffic per flop.
//
//   warp 9     TMA producer: Q_A, Q_B once; then K_0, V_0, K_1, V_1, ... through
//              one ring of NSLOT shared-memory slots (128-byte swizzle; rows
//              past the end arrive as zeros, like the pages' zero-filled
//              staging beyond kv_end)
//   warp 8     tcgen05 issuer (one thread), per KV tile j:
//                PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
//              S_X = Q_X K^T lands in TMEM (128 f32 columns per tile); the
//              softmax overwrites it in place with P_X (16-bit, 64 columns) and
//              O_X += P_X V reads P straight from TMEM (A-from-TMEM MMA form).
//              While the softmax of tile A works on S_A(j+1), the tensor core
//              runs PV_B(j) and S_B(j+1), and vice versa.
//   warps 0-3  softmax of tile A, warps 4-7 softmax of tile B: one thread per
//              query row == TMEM lane; mask only on diagonal / tail tiles; online
//              max / exp2 / sum; lazy O rescale in TMEM (only when the running
//              max grew by more than 2^8); P back to TMEM; finally O / l to
//              global memory.
//
// TMEM (512 columns): S_A | S_B | O_A | O_B.  Because every MMA of the CTA is
// issued by one thread and tcgen05 MMAs complete in issue order, S_X(j+1)
// (issued after PV_X(j)) never overwrites P_X(j) before PV_X(j) has read it,
// and when the softmax sees S_X(j+1) ready, PV_X(j) has finished -- so the O
// rescale never needs an extra wait.
//
// KV tiles entirely above the diagonal are never loaded (causal block skip),
// and the grid runs the longest query tiles first.  Every pipeline wait is
// bounded by a watchdog: a wait that does not complete records a code in
// g_fa_status, tells its CTA to stop, and the CTA drains its in-flight copies
// and MMAs, frees its TMEM and exits (no trap, no hang).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "fa_prefill.h"
#include "sm103_ptx.cuh"

namespace fa {

constexpr int BM = 128;           // query rows per tile == TMEM lanes == M of both MMAs
constexpr int BN = 128;           // keys per KV tile == N of S = Q K^T == K of P V
constexpr int NUM_THREADS = 384;  // warpgroups 0, 1: softmax of tiles A, B; warpgroup 2: MMA, producer
constexpr int MMA_WARP = 8;
constexpr int PRODUCER_WARP = 9;   // warps 10 and 11 only complete warpgroup 2
// Register budgets: launched at 168 per thread (65536 / 384, rounded down to
// a multiple of 8); warpgroup 2 gives registers back so the softmax
// warpgroups can hold a whole S row (128 f32) without spilling.
constexpr uint32_t LAUNCH_REGS = 168;
constexpr uint32_t REGS_SOFTMAX = 208;
constexpr uint32_t REGS_CONTROL = 56;
static_assert(128 * REGS_CONTROL + 256 * REGS_SOFTMAX <= NUM_THREADS * LAUNCH_REGS,
              "register split exceeds the launch allocation");
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_TAU = 8.0f;  // lazy rescale threshold in log2 units (P <= 2^8)
constexpr unsigned long long WATCHDOG_NS = 2000000000ull;  // 2 s per wait

// Watchdog codes (bits 0-7 of g_fa_status).
enum : uint32_t {
  WD_PRODUCER_EMPTY = 1,
  WD_MMA_Q = 3,
  WD_MMA_KV_FULL = 4,
  WD_MMA_P_FULL = 5,
  WD_SOFTMAX_S_FULL = 7,
  WD_SOFTMAX_O_DONE = 8,
  WD_DRAIN = 9,
};

// Shared-memory plan of one CTA, all offsets from a 1024-byte aligned base.
// The request is computed from this plan and nothing else, so the launcher
// cannot drift from the layout.
template <int HD>
struct Layout {
  static constexpr uint32_t KCH = HD / 64;           // 128-byte (64-element) column blocks along hd
  static constexpr uint32_t Q_BYTES = BM * HD * 2;   // one query tile
  static constexpr uint32_t SLOT_BYTES = BN * HD * 2;  // one K or one V tile
  static constexpr int NSLOT = HD == 128 ? 5 : 8;    // K/V ring depth (loads in flight)
  static constexpr uint32_t OFF_Q = 0;               // Q_A, Q_B
  static constexpr uint32_t OFF_RING = 2 * Q_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_RING + NSLOT * SLOT_BYTES;
  // q_full, full[NSLOT], empty[NSLOT], s_full[2], p_full[2], o_final, drain
  static constexpr uint32_t NUM_BARS = 1 + 2 * NSLOT + 2 + 2 + 2;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;  // [0] TMEM base, [1] abort flag
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static constexpr uint32_t REQUEST = BYTES + 1024;  // slack to align the dynamic base
  // TMEM columns: S_A | S_B | O_A | O_B (P_X overwrites the first BN/2 columns of S_X)
  static constexpr uint32_t TM_S = 0;
  static constexpr uint32_t TM_O = 2 * BN;
  static_assert(TM_O + 2 * HD <= TMEM_COLS, "TMEM plan");
  static_assert(OFF_RING % 1024 == 0 && SLOT_BYTES % 1024 == 0, "swizzle atoms");
};

struct Params {
  uint16_t* o;
  int B, Hq, Hkv, Sq, Skv;
  int G;           // Hq / Hkv
  int n_qtiles;    // ceil(Sq / BM)
  int pair_heads;  // 1: tiles A, B = query heads 2p, 2p+1 at the same rows; 0: rows 2t, 2t+1 of one head
  int causal;
  float sl2;       // scale * log2(e)
  unsigned long long watchdog_ns;
};

// The two query tiles of one CTA.  Longest tiles first; for head pairs the
// G/2 CTAs of one KV group are adjacent so their K/V tiles come from L2.
struct Work {
  int b, hk;
  int hq[2];
  int q0[2];
  bool has[2];
};

__device__ __forceinline__ Work decode_work(const Params& p) {
  Work w;
  if (p.pair_heads) {
    const int pairs = p.Hq / 2;
    const int per_qt = pairs * p.B;
    const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x / per_qt);
    const int rem = static_cast<int>(blockIdx.x % per_qt);
    w.b = rem / pairs;
    const int pi = rem % pairs;
    w.hq[0] = 2 * pi;
    w.hq[1] = 2 * pi + 1;
    w.q0[0] = w.q0[1] = qt * BM;
    w.has[0] = w.has[1] = true;
  } else {
    const int npq = (p.n_qtiles + 1) / 2;
    const int per = p.Hq * p.B;
    const int pq = npq - 1 - static_cast<int>(blockIdx.x / per);
    const int rem = static_cast<int>(blockIdx.x % per);
    w.b = rem / p.Hq;
    w.hq[0] = w.hq[1] = rem % p.Hq;
    w.q0[0] = 2 * pq * BM;
    w.q0[1] = w.q0[0] + BM;
    w.has[0] = true;
    w.has[1] = w.q0[1] < p.Sq;
  }
  w.hk = w.hq[0] / p.G;
  return w;
}

// KV tiles a query tile at rows [q0, q0 + BM) must visit (causal skip), and
// the number of keys every row of the tile sees (tiles below that need no mask).
__device__ __forceinline__ int kv_tiles(const Params& p, int q0, bool has) {
  if (!has) return 0;
  const int off = p.Skv - p.Sq;
  const int q_last = min(q0 + BM, p.Sq) - 1;
  const int kv_hi = p.causal ? min(p.Skv, off + q_last + 1) : p.Skv;
  return kv_hi > 0 ? (kv_hi + BN - 1) / BN : 0;
}

__device__ unsigned int g_fa_status = 0;

// Slow path of a bounded wait: poll, then give up after the watchdog limit
// (or as soon as another role of this CTA has given up).
__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                       unsigned long long limit_ns, uint32_t code) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1u;
      const uint32_t cta = blockIdx.x < 0xFFFFFFu ? blockIdx.x : 0xFFFFFFu;
      atomicCAS(&g_fa_status, 0u, (code & 0xFFu) | (cta << 8));
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         unsigned long long limit_ns, uint32_t code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, abort_flag, limit_ns, code);
}

// Warp-uniform bounded wait (all 32 lanes call it; all get the same answer).
__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity,
                                              volatile uint32_t* abort_flag,
                                              unsigned long long limit_ns, uint32_t code) {
  const bool ok = wait_bar(bar, parity, abort_flag, limit_ns, code);
  return __all_sync(0xffffffffu, ok);
}

// Drain wait used only on the abort path: bounded, ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > limit_ns) {
      atomicCAS(&g_fa_status, 0u, WD_DRAIN);
      return;
    }
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

template <int HD, bool BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fa_prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const Params p) {
  using L = Layout<HD>;
  constexpr int NSLOT = L::NSLOT;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);

  const uint32_t sQ = sbase + L::OFF_Q;
  const uint32_t sRing = sbase + L::OFF_RING;
  const uint32_t bar = sbase + L::OFF_BAR;
  const uint32_t bQ = bar;
  auto bFull = [&](int s) { return bar + 8u * (1 + s); };
  auto bEmpty = [&](int s) { return bar + 8u * (1 + NSLOT + s); };
  auto bSfull = [&](int x) { return bar + 8u * (1 + 2 * NSLOT + x); };
  auto bPfull = [&](int x) { return bar + 8u * (3 + 2 * NSLOT + x); };
  const uint32_t bOfinal = bar + 8u * (5 + 2 * NSLOT);
  const uint32_t bDrain = bar + 8u * (6 + 2 * NSLOT);
  uint32_t* misc = reinterpret_cast<uint32_t*>(gbase + L::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const Work w = decode_work(p);
  const int nA = kv_tiles(p, w.q0[0], w.has[0]);
  const int nB = kv_tiles(p, w.q0[1], w.has[1]);
  const int n = max(nA, nB);  // KV tiles the CTA streams; tile X uses the first n_X

  if (threadIdx.x == 0) {
    ptx::mbar_init(bQ, 1);
    for (int s = 0; s < NSLOT; ++s) {
      ptx::mbar_init(bFull(s), 1);
      ptx::mbar_init(bEmpty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(bSfull(x), 1);
      ptx::mbar_init(bPfull(x), BM);  // one arrival per softmax thread of tile x
    }
    ptx::mbar_init(bOfinal, 1);
    ptx::mbar_init(bDrain, 1);
    misc[1] = 0u;
    ptx::mbar_fence_init();
  }
  if (warp == MMA_WARP) {
    ptx::tmem_alloc(ptx::smem_u32(misc), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp >= MMA_WARP) {
  ptx::setmaxnreg_dec<REGS_CONTROL>();
  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      ptx::mbar_arrive_expect_tx(bQ, L::Q_BYTES * (w.has[1] ? 2u : 1u));
      for (int x = 0; x < 2; ++x) {
        if (!w.has[x]) continue;
#pragma unroll
        for (int c = 0; c < (int)L::KCH; ++c)
          ptx::tma_load_4d(sQ + x * L::Q_BYTES + c * (BM * 128), &tmQ, bQ, c * 64, w.hq[x], w.q0[x], w.b);
      }
      // loads in order K_0, V_0, K_1, V_1, ...; load i goes to slot i % NSLOT
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < 2 * n; ++i) {
        const int s = i % NSLOT;
        if (i >= NSLOT) ok = wait_bar(bEmpty(s), ((i / NSLOT) & 1) ^ 1u, abort_flag, p.watchdog_ns, WD_PRODUCER_EMPTY);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(bFull(s), L::SLOT_BYTES);
        const CUtensorMap* m = (i & 1) ? &tmV : &tmK;
#pragma unroll
        for (int c = 0; c < (int)L::KCH; ++c)
          ptx::tma_load_4d(sRing + s * L::SLOT_BYTES + c * (BN * 128), m, bFull(s), c * 64, w.hk, (i >> 1) * BN, w.b);
        ++issued;
      }
      if (!ok) {
        // abort: let every copy already issued land before the CTA exits
        drain_wait(bQ, 0, p.watchdog_ns);
        for (int s = 0; s < NSLOT && s < issued; ++s) {
          const int last = s + NSLOT * ((issued - 1 - s) / NSLOT);
          drain_wait(bFull(s), (last / NSLOT) & 1, p.watchdog_ns);
        }
      }
    }
  } else if (warp == MMA_WARP) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = ptx::idesc_f16(BF16, BM, BN, false, false);  // Q, K both K-major
      constexpr uint32_t IDESC_O = ptx::idesc_f16(BF16, BM, HD, false, true);   // P from TMEM, V MN-major
      auto issue_s = [&](int x, int slot) {
        const uint32_t d = tmem + L::TM_S + x * BN;
        const uint32_t q = sQ + x * L::Q_BYTES;
        const uint32_t k = sRing + slot * L::SLOT_BYTES;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t o = (kk / 4) * (BM * 128) + (kk % 4) * 32;
          ptx::mma_f16_ss(d, ptx::sdesc_sw128(q + o, 16, 1024), ptx::sdesc_sw128(k + o, 16, 1024), IDESC_S,
                          kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(bSfull(x));
      };
      auto issue_pv = [&](int x, int slot, bool acc) {
        const uint32_t d = tmem + L::TM_O + x * HD;
        const uint32_t a = tmem + L::TM_S + x * BN;  // P_X, 2 elements per column
        const uint32_t v = sRing + slot * L::SLOT_BYTES;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          ptx::mma_f16_ts(d, a + kk * 8, ptx::sdesc_sw128(v + kk * (16 * 128), BN * 128, 1024), IDESC_O,
                          (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = wait_bar(bQ, 0, abort_flag, p.watchdog_ns, WD_MMA_Q);
      if (ok && n > 0) {
        ok = wait_bar(bFull(0), 0, abort_flag, p.watchdog_ns, WD_MMA_KV_FULL);
        if (ok) {
          ptx::tc_fence_after();
          if (nA > 0) issue_s(0, 0);
          if (nB > 0) issue_s(1, 0);
          ptx::mma_commit(bEmpty(0));
        }
      }
      for (int j = 0; ok && j < n; ++j) {
        const int iv = 2 * j + 1, sv = iv % NSLOT;  // V_j
        const int ik = 2 * j + 2, sk = ik % NSLOT;  // K_{j+1}
        const bool more = j + 1 < n;
        ok = wait_bar(bFull(sv), (iv / NSLOT) & 1, abort_flag, p.watchdog_ns, WD_MMA_KV_FULL);
        if (!ok) break;
        if (more) {
          ok = wait_bar(bFull(sk), (ik / NSLOT) & 1, abort_flag, p.watchdog_ns, WD_MMA_KV_FULL);
          if (!ok) break;
        }
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const int nX = x == 0 ? nA : nB;
          if (j < nX) {
            ok = wait_bar(bPfull(x), j & 1, abort_flag, p.watchdog_ns, WD_MMA_P_FULL);
            if (!ok) break;
            ptx::tc_fence_after();
            issue_pv(x, sv, j > 0);
          }
          if (x == 1) ptx::mma_commit(bEmpty(sv));  // V_j no longer needed once PV_B(j) is done
          if (more && j + 1 < nX) issue_s(x, sk);
        }
        if (!ok) break;
        if (more) ptx::mma_commit(bEmpty(sk));
      }
      if (ok) {
        ptx::mma_commit(bOfinal);
      } else {
        ptx::mma_commit(bDrain);  // completes once every MMA issued above has finished
        drain_wait(bDrain, 0, p.watchdog_ns);
      }
    }
  }
  } else {
    ptx::setmaxnreg_inc<REGS_SOFTMAX>();
    // -------------------------------------------------------------- softmax
    const int x = warp >> 2;          // query tile of this warpgroup
    const int r = threadIdx.x & 127;  // row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + L::TM_S + x * BN;
    const uint32_t tO = tmem + lane_off + L::TM_O + x * HD;
    const int q0 = x == 0 ? w.q0[0] : w.q0[1];
    const int hqx = x == 0 ? w.hq[0] : w.hq[1];
    const bool hasx = x == 0 ? w.has[0] : w.has[1];
    const int nX = x == 0 ? nA : nB;
    const int off = p.Skv - p.Sq;
    const int kv_all = p.causal ? min(p.Skv, off + q0 + 1) : p.Skv;       // keys every row sees
    const int row_lim = p.causal ? min(p.Skv, off + q0 + r + 1) : p.Skv;  // keys this row sees
    const float sl2 = p.sl2;
    float m_ref = -INFINITY;  // running max (log2 domain) that O and l are scaled to
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < nX; ++j) {
      ok = warp_wait_bar(bSfull(x), j & 1, abort_flag, p.watchdog_ns, WD_SOFTMAX_S_FULL);
      if (!ok) break;
      ptx::tc_fence_after();
      uint32_t sr[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) ptx::tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
      ptx::tmem_wait_ld();
      ptx::reg_fence(sr);
      float s[BN];
#pragma unroll
      for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(sr[c]);
      const int kv0 = j * BN;
      if (kv0 + BN > kv_all) {  // diagonal or tail tile: mask per element
        const int lim = row_lim - kv0;
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= lim) s[c] = -INFINITY;
      }
      // row max: eight independent 3-input max chains, then combine
      float mk[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mk[k] = ptx::fmax3(s[k], s[8 + k], s[16 + k]);
#pragma unroll
      for (int t = 3; t < 15; t += 2)
#pragma unroll
        for (int k = 0; k < 8; ++k) mk[k] = ptx::fmax3(mk[k], s[8 * t + k], s[8 * t + 8 + k]);
#pragma unroll
      for (int k = 0; k < 8; ++k) mk[k] = fmaxf(mk[k], s[120 + k]);
      const float mx = ptx::fmax3(ptx::fmax3(mk[0], mk[1], mk[2]), ptx::fmax3(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7]));
      const float m_new = fmaxf(m_ref, mx * sl2);
      const bool resc = m_new > m_ref + RESCALE_TAU;  // -inf -> finite always rescales
      float alpha = 1.f;
      if (resc) {
        alpha = ptx::ex2(m_ref - m_new);  // 0 when m_ref == -inf
        m_ref = m_new;
        l *= alpha;
      }
      const float mb = (m_ref == -INFINITY) ? 0.f : m_ref;
      // p = 2^(s * scale * log2e - m): packed FMA, ex2 per element, the row sum
      // in four packed partial sums, and P packed to 16-bit pairs
      const uint64_t c2 = ptx::pk(sl2, sl2);
      const uint64_t nb2 = ptx::pk(-mb, -mb);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
      uint32_t pp[BN / 2];
#pragma unroll
      for (int c = 0; c < BN; c += 2) {
        float x0, x1;
        ptx::upk(ptx::fma2(ptx::pk(s[c], s[c + 1]), c2, nb2), x0, x1);
        const float e0 = ptx::ex2(x0), e1 = ptx::ex2(x1);
        acc[(c >> 1) & 3] = ptx::add2(acc[(c >> 1) & 3], ptx::pk(e0, e1));
        pp[c >> 1] = pack2<BF16>(e0, e1);
      }
      {
        float a0, a1;
        ptx::upk(ptx::add2(ptx::add2(acc[0], acc[1]), ptx::add2(acc[2], acc[3])), a0, a1);
        l += a0 + a1;
      }
      // the running max moved: rescale O_X in TMEM (PV_X(j-1) finished before S_X(j) did)
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        const uint64_t a2 = ptx::pk(alpha, alpha);
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t orr[32];
          ptx::tmem_ld32(tO + c * 32, orr);
          ptx::tmem_wait_ld();
          ptx::reg_fence(orr);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float o0, o1;
            ptx::upk(ptx::mul2(ptx::pk(__uint_as_float(orr[e]), __uint_as_float(orr[e + 1])), a2), o0, o1);
            orr[e] = __float_as_uint(o0);
            orr[e + 1] = __float_as_uint(o1);
          }
          ptx::tmem_st32(tO + c * 32, orr);
        }
      }
      // P_X over the first BN/2 columns of S_X
      ptx::tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pp[0]));
      ptx::tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pp[32]));
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bPfull(x));
    }
    // ------------------------------------------------------------ epilogue
    if (ok && nX > 0) {
      ok = warp_wait_bar(bOfinal, 0, abort_flag, p.watchdog_ns, WD_SOFTMAX_O_DONE);
      if (ok) ptx::tc_fence_after();
    }
    if (ok && hasx) {
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const int qrow = q0 + r;
      const bool row_ok = qrow < p.Sq;
      uint4* dst =
          reinterpret_cast<uint4*>(p.o + ((static_cast<size_t>(w.b) * p.Sq + qrow) * p.Hq + hqx) * HD);
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t orr[32];
        if (nX > 0) {
          ptx::tmem_ld32(tO + c * 32, orr);
          ptx::tmem_wait_ld();
          ptx::reg_fence(orr);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = 0u;
        }
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 v;
            v.x = pack2<BF16>(__uint_as_float(orr[8 * e + 0]) * inv_l, __uint_as_float(orr[8 * e + 1]) * inv_l);
            v.y = pack2<BF16>(__uint_as_float(orr[8 * e + 2]) * inv_l, __uint_as_float(orr[8 * e + 3]) * inv_l);
            v.z = pack2<BF16>(__uint_as_float(orr[8 * e + 4]) * inv_l, __uint_as_float(orr[8 * e + 5]) * inv_l);
            v.w = pack2<BF16>(__uint_as_float(orr[8 * e + 6]) * inv_l, __uint_as_float(orr[8 * e + 7]) * inv_l);
            dst[c * 4 + e] = v;
          }
        }
      }
    }
  }

  // ---- teardown: every role is done (or has drained); free TMEM
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// =============================================================== host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encoder() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load();
  if (f) return f;
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || ptr == nullptr) {
    (void)cudaGetLastError();
    return nullptr;
  }
  f = reinterpret_cast<EncodeTiledFn>(ptr);
  fn.store(f);
  return f;
}

// 4-D map over a BSHD tensor: dims (hd, H, S, B), box (64, 1, 128, 1), 128-byte swizzle.
static bool encode_bshd(CUtensorMap* m, EncodeTiledFn enc, const void* base, bool bf16, int B, int S, int H, int hd) {
  const cuuint64_t dims[4] = {(cuuint64_t)hd, (cuuint64_t)H, (cuuint64_t)(S > 0 ? S : 1), (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)hd * 2, (cuuint64_t)H * hd * 2, (cuuint64_t)(S > 0 ? S : 1) * H * hd * 2};
  const cuuint32_t box[4] = {64, 1, 128, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// CTAs of one launch: each CTA takes two 128-row query tiles sharing one KV head.
static long long grid_size(int B, int Hq, int Hkv, int Sq) {
  const long long n_qt = (Sq + BM - 1) / BM;
  if ((Hq / Hkv) % 2 == 0) return n_qt * (Hq / 2) * B;
  return ((n_qt + 1) / 2) * Hq * (long long)B;
}

constexpr int MAX_DEVICES = 64;

// Per-device facts, filled once: 1 = sm_103 with enough opt-in shared memory.
static std::atomic<int> g_dev_ok[MAX_DEVICES];
static std::atomic<int> g_attr_set[MAX_DEVICES][4];

static int check_device(int* dev_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
    (void)cudaGetLastError();
    return FA_ERR_DEVICE;
  }
  *dev_out = dev;
  int st = g_dev_ok[dev].load();
  if (st == 0) {
    int major = 0, minor = 0, optin = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      return FA_ERR_DEVICE;
    }
    if (major != 10 || minor != 3) st = -FA_ERR_DEVICE;
    else if ((unsigned)optin < Layout<128>::REQUEST) st = -FA_ERR_SMEM;
    else st = 1;
    g_dev_ok[dev].store(st);
  }
  return st == 1 ? FA_OK : -st;
}

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na > 0 && nb > 0 && x < y + nb && y < x + na;
}

template <int HD, bool BF16>
static int launch(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int Sq, int Skv,
                  int causal, float scale, cudaStream_t stream, int dev) {
  using L = Layout<HD>;
  auto kern = fa_prefill_kernel<HD, BF16>;
  const int slot = (HD == 128 ? 2 : 0) + (BF16 ? 1 : 0);
  if (g_attr_set[dev][slot].load() == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::REQUEST) != cudaSuccess) {
      (void)cudaGetLastError();
      return FA_ERR_SMEM;
    }
    g_attr_set[dev][slot].store(1);
  }
  EncodeTiledFn enc = encoder();
  if (!enc) return FA_ERR_LAUNCH;
  CUtensorMap mq, mk, mv;
  if (!encode_bshd(&mq, enc, q, BF16, B, Sq, Hq, HD) || !encode_bshd(&mk, enc, k, BF16, B, Skv, Hkv, HD) ||
      !encode_bshd(&mv, enc, v, BF16, B, Skv, Hkv, HD))
    return FA_ERR_LAUNCH;
  Params prm;
  prm.o = static_cast<uint16_t*>(o);
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Sq = Sq;
  prm.Skv = Skv;
  prm.G = Hq / Hkv;
  prm.n_qtiles = (Sq + BM - 1) / BM;
  prm.pair_heads = (prm.G % 2 == 0) ? 1 : 0;
  prm.causal = causal ? 1 : 0;
  prm.sl2 = scale * 1.4426950408889634f;
  prm.watchdog_ns = WATCHDOG_NS;
  const long long grid = grid_size(B, Hq, Hkv, Sq);
  kern<<<dim3((unsigned)grid), dim3(NUM_THREADS), L::REQUEST, stream>>>(mq, mk, mv, prm);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  return FA_OK;
}

static int run(bool bf16, const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int Sq,
               int Skv, int hd, int causal, float scale, void* stream) {
  if (B < 0 || Sq < 0 || Skv < 0 || Hq < 1 || Hkv < 1) return FA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (hd != 64 && hd != 128) return FA_ERR_UNSUPPORTED;
  if (B == 0 || Sq == 0) return FA_OK;  // nothing to compute; no pointer is read
  if (!q || !o) return FA_ERR_INVALID_ARG;
  if (Skv > 0 && (!k || !v)) return FA_ERR_INVALID_ARG;
  if (Skv == 0) k = v = q;  // no key is ever loaded; the K/V maps only need a valid base
  const auto mis = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) != 0; };
  if (mis(q) || mis(k) || mis(v) || mis(o)) return FA_ERR_ALIGNMENT;
  // TMA coordinates are 32-bit and a box may start up to 127 rows past the end.
  const long long lim = 0x7FFFFFFFLL - 256;
  if ((long long)Sq > lim || (long long)Skv > lim) return FA_ERR_UNSUPPORTED;
  const unsigned long long qn = (unsigned long long)B * Sq * Hq * hd;
  const unsigned long long kn = (unsigned long long)B * Skv * Hkv * hd;
  if ((unsigned long long)Sq * Hq * hd * 2 >= (1ull << 40) || (unsigned long long)Skv * Hkv * hd * 2 >= (1ull << 40))
    return FA_ERR_UNSUPPORTED;
  if (overlaps(o, qn * 2, q, qn * 2) || overlaps(o, qn * 2, k, kn * 2) || overlaps(o, qn * 2, v, kn * 2))
    return FA_ERR_INVALID_ARG;
  if (grid_size(B, Hq, Hkv, Sq) > 0x7FFFFFFFLL) return FA_ERR_UNSUPPORTED;
  int dev = -1;
  const int ds = check_device(&dev);
  if (ds != FA_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (hd == 128)
    return bf16 ? launch<128, true>(q, k, v, o, B, Hq, Hkv, Sq, Skv, causal, scale, st, dev)
                : launch<128, false>(q, k, v, o, B, Hq, Hkv, Sq, Skv, causal, scale, st, dev);
  return bf16 ? launch<64, true>(q, k, v, o, B, Hq, Hkv, Sq, Skv, causal, scale, st, dev)
              : launch<64, false>(q, k, v, o, B, Hq, Hkv, Sq, Skv, causal, scale, st, dev);
}

}  // namespace fa

// ================================================================== C ABI

extern "C" int fa_prefill(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int Sq,
                          int Skv, int hd, int causal, float scale, void* stream) {
  return fa::run(false, q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, causal, scale, stream);
}

extern "C" int fa_prefill_bf16(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int Sq,
                               int Skv, int hd, int causal, float scale, void* stream) {
  return fa::run(true, q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, causal, scale, stream);
}

extern "C" const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null pointer, bad size, Hq % Hkv != 0, bad scale or aliasing";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: hd must be 64 or 128 and tensors must fit TMA coordinates";
    case FA_ERR_ALIGNMENT: return "FA_ERR_ALIGNMENT: q, k, v and o must be 16-byte aligned";
    case FA_ERR_SMEM: return "FA_ERR_SMEM: shared-memory request does not fit the device";
    case FA_ERR_LAUNCH: return "FA_ERR_LAUNCH: TMA descriptor encode or kernel launch failed";
    case FA_ERR_DEVICE: return "FA_ERR_DEVICE: no current device or not an sm_103 GPU";
    default: return "unknown fa_status_t";
  }
}

extern "C" unsigned int fa_smem_bytes(int hd) {
  if (hd == 128) return fa::Layout<128>::REQUEST;
  if (hd == 64) return fa::Layout<64>::REQUEST;
  return 0u;
}

extern "C" int fa_debug_status(void) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, fa::g_fa_status, sizeof(v)) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  return static_cast<int>(v);
}

extern "C" int fa_debug_status_clear(void) {
  const unsigned int z = 0;
  if (cudaMemcpyToSymbol(fa::g_fa_status, &z, sizeof(z)) != cudaSuccess) {
    (void)cudaGetLastError();
    return FA_ERR_DEVICE;
  }
  return FA_OK;
}
