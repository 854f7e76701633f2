// fa_prefill.cu -- causal prefill flash attention for GB300 (sm_103a).
//
//   O = softmax(scale * Q K^T + causal mask) V,  16-bit Q/K/V/O, f32 accumulate.
//
// One CTA owns one 128-row query tile of one (batch, query head) and walks the
// KV tiles that tile can see, keeping the running row max m and row sum l of
// the online softmax (minfer "53 · r50 — FA_TKV 32->16 occupancy experiment",
// section 2: stage K/V, S = Q K^T, mask, max, exp, sum, rescale O, O += P V).
// The pages' kernel does this with wmma fragments and cp.async on another GPU;
// here every stage is re-planned for Blackwell:
//
//   warp 4  TMA producer: Q once, then K_j and V_j into a 2-stage mbarrier ring
//           (out-of-range rows arrive as zeros, like the pages' zero-filled
//           staging beyond kv_end)
//   warp 5  tcgen05 issuer (one thread): S_j = Q K_j^T into one of two TMEM
//           S buffers, and O += P_j V_j into a TMEM O accumulator
//   warps 0-3  softmax: one thread per query row == TMEM lane; load S_j from
//           TMEM, apply the causal/tail mask only on tiles that need it, online
//           max / exp2 / sum, lazy O rescale in TMEM, write P_j (16-bit) into a
//           128-byte-swizzled shared tile that the P V MMA reads; finally O / l
//           to global memory
//
// KV tiles entirely above the diagonal are never loaded (causal block skip),
// and the grid is ordered longest query tile first.  Every pipeline wait is
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
constexpr int NSTAGE = 2;         // depth of the K ring and of the V ring
constexpr int NUM_THREADS = 192;  // warps 0-3 softmax, 4 producer, 5 MMA
constexpr int PRODUCER_WARP = 4;
constexpr int MMA_WARP = 5;
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_TAU = 8.0f;  // lazy rescale threshold in log2 units (P <= 2^8)
constexpr unsigned long long WATCHDOG_NS = 2000000000ull;  // 2 s per wait

// Watchdog codes (bits 0-7 of g_fa_status).
enum : uint32_t {
  WD_PRODUCER_K_EMPTY = 1,
  WD_PRODUCER_V_EMPTY = 2,
  WD_MMA_Q = 3,
  WD_MMA_K_FULL = 4,
  WD_MMA_P_FULL = 5,
  WD_MMA_V_FULL = 6,
  WD_SOFTMAX_S_FULL = 7,
  WD_SOFTMAX_O_DONE = 8,
  WD_DRAIN = 9,
};

// Shared-memory plan of one CTA, all offsets from a 1024-byte aligned base.
// The request is computed from this plan and nothing else, so the launcher
// cannot drift from the layout.
template <int HD>
struct Layout {
  static constexpr uint32_t KCH = HD / 64;         // 128-byte (64-element) column blocks along hd
  static constexpr uint32_t Q_BYTES = BM * HD * 2;
  static constexpr uint32_t KV_BYTES = BN * HD * 2;
  static constexpr uint32_t P_BYTES = BM * BN * 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + NSTAGE * KV_BYTES;
  static constexpr uint32_t OFF_P = OFF_V + NSTAGE * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_P + P_BYTES;
  // q_full, k_full[NS], k_empty[NS], v_full[NS], v_empty[NS], s_full[2], p_full, o_done, drain
  static constexpr uint32_t NUM_BARS = 1 + 4 * NSTAGE + 2 + 3;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;  // [0] TMEM base, [1] abort flag
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static constexpr uint32_t REQUEST = BYTES + 1024;  // slack to align the dynamic base
  // TMEM columns: S0 | S1 | O
  static constexpr uint32_t TM_S0 = 0;
  static constexpr uint32_t TM_O = 2 * BN;
  static_assert(TM_O + HD <= TMEM_COLS, "TMEM plan");
  static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && OFF_P % 1024 == 0, "swizzle atoms");
};

struct Params {
  uint16_t* o;
  int B, Hq, Hkv, Sq, Skv;
  int G;         // Hq / Hkv
  int n_qtiles;  // ceil(Sq / BM)
  int causal;
  float sl2;     // scale * log2(e)
  unsigned long long watchdog_ns;
};

__device__ unsigned int g_fa_status = 0;

// Slow path of a bounded wait: poll, then give up after the watchdog limit
// (or as soon as another role of this CTA has given up).
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
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
__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
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
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);

  const uint32_t sQ = sbase + L::OFF_Q;
  const uint32_t sK = sbase + L::OFF_K;
  const uint32_t sV = sbase + L::OFF_V;
  const uint32_t sP = sbase + L::OFF_P;
  const uint32_t bar = sbase + L::OFF_BAR;
  const uint32_t bQ = bar;
  auto bKfull = [&](int s) { return bar + 8u * (1 + s); };
  auto bKempty = [&](int s) { return bar + 8u * (1 + NSTAGE + s); };
  auto bVfull = [&](int s) { return bar + 8u * (1 + 2 * NSTAGE + s); };
  auto bVempty = [&](int s) { return bar + 8u * (1 + 3 * NSTAGE + s); };
  auto bSfull = [&](int x) { return bar + 8u * (1 + 4 * NSTAGE + x); };
  const uint32_t bPfull = bar + 8u * (3 + 4 * NSTAGE);
  const uint32_t bOdone = bar + 8u * (4 + 4 * NSTAGE);
  const uint32_t bDrain = bar + 8u * (5 + 4 * NSTAGE);
  uint32_t* misc = reinterpret_cast<uint32_t*>(gbase + L::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- which tile: longest query tiles first; the G query heads that share a
  // KV head are adjacent so their K/V tiles are reused from L2.
  const int per_qt = p.Hq * p.B;
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x / per_qt);
  const int rem = static_cast<int>(blockIdx.x % per_qt);
  const int b = rem / p.Hq;
  const int hq = rem % p.Hq;
  const int hk = hq / p.G;
  const int q0 = qt * BM;
  // Causal geometry, bottom-right aligned: row i sees keys j <= off + i.
  const int off = p.Skv - p.Sq;
  const int q_last = min(q0 + BM, p.Sq) - 1;
  const int kv_hi = p.causal ? min(p.Skv, off + q_last + 1) : p.Skv;   // keys any row sees
  const int n_kv = kv_hi > 0 ? (kv_hi + BN - 1) / BN : 0;              // tiles above the diagonal skipped
  const int kv_all = p.causal ? min(p.Skv, off + q0 + 1) : p.Skv;      // keys every row sees

  if (threadIdx.x == 0) {
    ptx::mbar_init(bQ, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      ptx::mbar_init(bKfull(s), 1);
      ptx::mbar_init(bKempty(s), 1);
      ptx::mbar_init(bVfull(s), 1);
      ptx::mbar_init(bVempty(s), 1);
    }
    ptx::mbar_init(bSfull(0), 1);
    ptx::mbar_init(bSfull(1), 1);
    ptx::mbar_init(bPfull, BM);  // one arrival per softmax thread
    ptx::mbar_init(bOdone, 1);
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

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      ptx::mbar_arrive_expect_tx(bQ, L::Q_BYTES);
#pragma unroll
      for (int c = 0; c < (int)L::KCH; ++c)
        ptx::tma_load_4d(sQ + c * (BM * 128), &tmQ, bQ, c * 64, hq, q0, b);
      int nk = 0, nv = 0;  // loads issued
      bool ok = true;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % NSTAGE;
        const uint32_t ph = (j / NSTAGE) & 1;
        if (j >= NSTAGE) ok = wait_bar(bKempty(s), ph ^ 1u, abort_flag, p.watchdog_ns, WD_PRODUCER_K_EMPTY);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(bKfull(s), L::KV_BYTES);
#pragma unroll
        for (int c = 0; c < (int)L::KCH; ++c)
          ptx::tma_load_4d(sK + s * L::KV_BYTES + c * (BN * 128), &tmK, bKfull(s), c * 64, hk, j * BN, b);
        ++nk;
        if (j >= NSTAGE) ok = wait_bar(bVempty(s), ph ^ 1u, abort_flag, p.watchdog_ns, WD_PRODUCER_V_EMPTY);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(bVfull(s), L::KV_BYTES);
#pragma unroll
        for (int c = 0; c < (int)L::KCH; ++c)
          ptx::tma_load_4d(sV + s * L::KV_BYTES + c * (BN * 128), &tmV, bVfull(s), c * 64, hk, j * BN, b);
        ++nv;
      }
      if (!ok) {
        // abort: let every copy already issued land before the CTA exits
        drain_wait(bQ, 0, p.watchdog_ns);
        for (int s = 0; s < NSTAGE; ++s) {
          // tiles s, s + NSTAGE, ... went to stage s; wait for the last one issued
          if (nk > s) {
            const int jk = s + NSTAGE * ((nk - 1 - s) / NSTAGE);
            drain_wait(bKfull(s), (jk / NSTAGE) & 1, p.watchdog_ns);
          }
          if (nv > s) {
            const int jv = s + NSTAGE * ((nv - 1 - s) / NSTAGE);
            drain_wait(bVfull(s), (jv / NSTAGE) & 1, p.watchdog_ns);
          }
        }
      }
    }
  } else if (warp == MMA_WARP) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = ptx::idesc_f16(BF16, BM, BN, false, false);  // Q, K both K-major
      constexpr uint32_t IDESC_O = ptx::idesc_f16(BF16, BM, HD, false, true);   // P K-major, V MN-major
      bool ok = wait_bar(bQ, 0, abort_flag, p.watchdog_ns, WD_MMA_Q);
      auto issue_s = [&](int j) {
        const int s = j % NSTAGE;
        const uint32_t d = tmem + L::TM_S0 + (j & 1) * BN;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint64_t a = ptx::sdesc_sw128(sQ + (kk / 4) * (BM * 128) + (kk % 4) * 32, 16, 1024);
          const uint64_t bd =
              ptx::sdesc_sw128(sK + s * L::KV_BYTES + (kk / 4) * (BN * 128) + (kk % 4) * 32, 16, 1024);
          ptx::mma_f16_ss(d, a, bd, IDESC_S, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(bSfull(j & 1));
        ptx::mma_commit(bKempty(s));
      };
      if (ok && n_kv > 0) {
        ok = wait_bar(bKfull(0), 0, abort_flag, p.watchdog_ns, WD_MMA_K_FULL);
        if (ok) {
          ptx::tc_fence_after();
          issue_s(0);
        }
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv) {
          const int s1 = (j + 1) % NSTAGE;
          ok = wait_bar(bKfull(s1), ((j + 1) / NSTAGE) & 1, abort_flag, p.watchdog_ns, WD_MMA_K_FULL);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_s(j + 1);
        }
        ok = wait_bar(bPfull, j & 1, abort_flag, p.watchdog_ns, WD_MMA_P_FULL);
        if (!ok) break;
        const int s = j % NSTAGE;
        ok = wait_bar(bVfull(s), (j / NSTAGE) & 1, abort_flag, p.watchdog_ns, WD_MMA_V_FULL);
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t a = ptx::sdesc_sw128(sP + (kk / 4) * (BM * 128) + (kk % 4) * 32, 16, 1024);
          const uint64_t bd = ptx::sdesc_sw128(sV + s * L::KV_BYTES + kk * (16 * 128), BN * 128, 1024);
          ptx::mma_f16_ss(tmem + L::TM_O, a, bd, IDESC_O, (j > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::mma_commit(bOdone);
        ptx::mma_commit(bVempty(s));
      }
      if (!ok) {
        ptx::mma_commit(bDrain);  // completes once every MMA issued above has finished
        drain_wait(bDrain, 0, p.watchdog_ns);
      }
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int r = threadIdx.x;  // row in the tile == TMEM lane
    const uint32_t t_row = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int row_lim = p.causal ? min(p.Skv, off + q0 + r + 1) : p.Skv;  // keys this row sees
    const float sl2 = p.sl2;
    float m_ref = -INFINITY;  // running max (log2 domain) that O and l are scaled to
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      ok = warp_wait_bar(bSfull(j & 1), (j >> 1) & 1, abort_flag, p.watchdog_ns, WD_SOFTMAX_S_FULL);
      if (!ok) break;
      ptx::tc_fence_after();
      uint32_t sr[BN];
      const uint32_t t_s = t_row + L::TM_S0 + (j & 1) * BN;
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) ptx::tmem_ld32(t_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
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
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < BN; ++c) mx = fmaxf(mx, s[c]);
      const float m_new = fmaxf(m_ref, mx * sl2);
      const bool resc = m_new > m_ref + RESCALE_TAU;  // -inf -> finite always rescales
      float alpha = 1.f;
      if (resc) {
        alpha = ptx::ex2(m_ref - m_new);  // 0 when m_ref == -inf
        m_ref = m_new;
        l *= alpha;
      }
      const float mb = (m_ref == -INFINITY) ? 0.f : m_ref;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < BN; ++c) {
        s[c] = ptx::ex2(fmaf(s[c], sl2, -mb));
        rs += s[c];
      }
      l += rs;
      // P V of the previous tile must be done before P is overwritten and O rescaled
      if (j > 0) {
        ok = warp_wait_bar(bOdone, (j - 1) & 1, abort_flag, p.watchdog_ns, WD_SOFTMAX_O_DONE);
        if (!ok) break;
        ptx::tc_fence_after();
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t orr[32];
            ptx::tmem_ld32(t_row + L::TM_O + c * 32, orr);
            ptx::tmem_wait_ld();
            ptx::reg_fence(orr);
#pragma unroll
            for (int x = 0; x < 32; ++x) orr[x] = __float_as_uint(__uint_as_float(orr[x]) * alpha);
            ptx::tmem_st32(t_row + L::TM_O + c * 32, orr);
          }
          ptx::tmem_wait_st();
        }
      }
      // P row -> 16-bit, K-major tile in the 128-byte swizzle layout the MMA reads
      const uint32_t prow = sP + r * 128;
#pragma unroll
      for (int g = 0; g < BN / 8; ++g) {
        const uint32_t addr = prow + (g / 8) * (BM * 128) + (((g % 8) ^ (r % 8)) * 16);
        ptx::st_shared_v4(addr, pack2<BF16>(s[g * 8 + 0], s[g * 8 + 1]), pack2<BF16>(s[g * 8 + 2], s[g * 8 + 3]),
                          pack2<BF16>(s[g * 8 + 4], s[g * 8 + 5]), pack2<BF16>(s[g * 8 + 6], s[g * 8 + 7]));
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bPfull);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && n_kv > 0) {
      ok = warp_wait_bar(bOdone, (n_kv - 1) & 1, abort_flag, p.watchdog_ns, WD_SOFTMAX_O_DONE);
      if (ok) ptx::tc_fence_after();
    }
    if (ok) {
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const int qrow = q0 + r;
      const bool row_ok = qrow < p.Sq;
      uint4* dst = reinterpret_cast<uint4*>(p.o + ((static_cast<size_t>(b) * p.Sq + qrow) * p.Hq + hq) * HD);
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t orr[32];
        if (n_kv > 0) {
          ptx::tmem_ld32(t_row + L::TM_O + c * 32, orr);
          ptx::tmem_wait_ld();
          ptx::reg_fence(orr);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) orr[x] = 0u;
        }
        if (row_ok) {
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            uint4 v;
            v.x = pack2<BF16>(__uint_as_float(orr[8 * x + 0]) * inv_l, __uint_as_float(orr[8 * x + 1]) * inv_l);
            v.y = pack2<BF16>(__uint_as_float(orr[8 * x + 2]) * inv_l, __uint_as_float(orr[8 * x + 3]) * inv_l);
            v.z = pack2<BF16>(__uint_as_float(orr[8 * x + 4]) * inv_l, __uint_as_float(orr[8 * x + 5]) * inv_l);
            v.w = pack2<BF16>(__uint_as_float(orr[8 * x + 6]) * inv_l, __uint_as_float(orr[8 * x + 7]) * inv_l);
            dst[c * 4 + x] = v;
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
  prm.causal = causal ? 1 : 0;
  prm.sl2 = scale * 1.4426950408889634f;
  prm.watchdog_ns = WATCHDOG_NS;
  const long long grid = (long long)prm.n_qtiles * Hq * B;
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
  const long long grid = (long long)((Sq + BM - 1) / BM) * Hq * B;
  if (grid > 0x7FFFFFFFLL) return FA_ERR_UNSUPPORTED;
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
