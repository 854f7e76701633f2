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
//              max grew by more than 2^8); P back to TMEM; finally O / l,
//              staged 128-byte swizzled in a ring slot the finished tile no
//              longer needs and written out by TMA tensor stores.
//
// TMEM (512 columns): S_A | S_B | O_A | O_B.  Because every MMA of the CTA is
// issued by one thread and tcgen05 MMAs complete in issue order, S_X(j+1)
// (issued after PV_X(j)) never overwrites P_X(j) before PV_X(j) has read it,
// and when the softmax sees S_X(j+1) ready, PV_X(j) has finished -- so the O
// rescale never needs an extra wait.
//
// KV tiles entirely above the diagonal are never loaded (causal block skip),
// and the grid runs the longest query tiles first.  The producer can also read
// K/V through a block table (paged cache) or from a cache whose capacity
// exceeds its valid length; only its TMA coordinates change.  Every pipeline
// wait is bounded by a watchdog: a wait that does not complete records a code
// in g_fa_status, tells its CTA to stop, and the CTA drains its in-flight
// copies and MMAs, frees its TMEM and exits (no trap, no hang).  Launches use
// programmatic dependent launch: set-up overlaps the previous kernel's tail,
// global memory is touched only after griddepcontrol.wait.
//
// The same translation unit holds the other kernels of the library, which
// share these helpers: the hd <= 64 kernel with S and P in separate TMEM
// columns (fa_prefill64.cuh), the hd = 256 kernel (fa_prefill256.cuh), the
// split-KV kernel for one piece per CTA (fa_prefill_sk_kernel, below) and its
// merge, the persistent kernel that runs split-KV schedules with several
// segments per CTA (fa_persistent.cuh), the opt-in kernel on CTA pairs
// (fa_prefill_pair.cuh) and the K/V-cache append (kv_append.cuh).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

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
constexpr unsigned long long WATCHDOG_NS = 2000000000ull;  // 2 s per wait (the default; see fa_debug_set_watchdog_ns)
// Drains wait for work already issued (TMA copies, MMAs), which always
// completes: their limit is fixed, whatever the wait limit.
constexpr unsigned long long DRAIN_NS = 2000000000ull;

// Watchdog codes (bits 0-7 of g_fa_status).
enum : uint32_t {
  WD_PRODUCER_EMPTY = 1,
  WD_MMA_Q = 3,
  WD_MMA_KV_FULL = 4,
  WD_MMA_P_FULL = 5,
  WD_SOFTMAX_S_FULL = 7,
  WD_SOFTMAX_O_DONE = 8,
  WD_DRAIN = 9,
  WD_PIECE_SLOT = 12,  // a split piece without a workspace slot (inconsistent schedule)
  WD_PAGE_BLOCK = 33,  // a block-table entry outside the pool (its tiles load as zeros)
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
  // q_full (Q and K_0), pair[NPB <= NSLOT] (V_j, K_j+1), empty[NSLOT] (hd 128: pair-empty, NPE of them),
  // s_full[2], p_full[2], o_final, drain
  static constexpr uint32_t NUM_BARS = 1 + 2 * NSLOT + 2 + 2 + 2;
  // [0] TMEM base, [1] abort flag, [2], [3] barrier and phase of tile A's early o_final (0: none)
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static constexpr uint32_t REQUEST = BYTES + 1024;  // slack to align the dynamic base
  // TMEM columns: S_A | S_B | O_A | O_B (P_X overwrites the first BN/2 columns of S_X)
  static constexpr uint32_t TM_S = 0;
  static constexpr uint32_t TM_O = 2 * BN;
  static_assert(TM_O + 2 * HD <= TMEM_COLS, "TMEM plan");
  static_assert(OFF_RING % 1024 == 0 && SLOT_BYTES % 1024 == 0, "swizzle atoms");
  static_assert(SLOT_BYTES == BM * HD * 2 && NSLOT >= 2, "each O tile is staged in a ring slot");
};

struct Params {
  uint16_t* o;
  int B, Hq, Hkv, Sq, Skv;
  int G;           // Hq / Hkv
  int n_qtiles;    // ceil(Sq / BM)
  int pair_heads;  // 1: tiles A, B = query heads 2p, 2p+1 at the same rows; 0: two adjacent row tiles of one head
  int lone_first;  // row tiles, odd tile count: 1 = tile 0 without a partner, 0 = the last tile (pair_first_tile)
  int causal;
  float sl2;       // scale * log2(e)
  unsigned long long watchdog_ns;
  // paged K/V (one-shot kernel only): K/V tile t of sequence b lives in pool
  // block block_table[b * max_pages + t * BN / page_size], rows from
  // (t * BN) % page_size; the last page is read through the tail maps
  const int* block_table;  // nullptr: contiguous [B][Skv][Hkv][hd] K/V
  int page_size, max_pages, num_blocks, last_page;
  float* lse;  // nullptr, or [B][Hq][Sq]: log sum_j exp(scale s_j) of every row (-inf: no key)
  int hd;      // head dimension of the tensors (<= the kernel's HD: the maps zero-fill and clip the rest)
};

// A row's log-sum-exp from the online-softmax state: m (log2 units of
// scale * log2(e) * s) and l = sum 2^(s' - m), so lse = (m + log2 l) ln 2.
__device__ __forceinline__ float row_lse(float m, float l) {
  return l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
}

// The two query tiles of one CTA.  Longest tiles first; for head pairs the
// G/2 CTAs of one KV group are adjacent so their K/V tiles come from L2.
struct Work {
  int b, hk;
  int hq[2];
  int q0[2];
  bool has[2];
};

// First query tile of row pair pq (MHA and odd GQA groups: one head, two
// adjacent 128-row tiles per CTA).  An even tile count pairs (2 pq, 2 pq + 1).
// An odd one leaves one tile without a partner: the last (pairs (2 pq,
// 2 pq + 1), tile B missing at the last pq) or, with lone_first, tile 0
// (tile 0 alone at pq = 0, then (2 pq - 1, 2 pq)).  Under the causal mask the
// last tile sees the most keys and tile 0 the fewest; the host picks the
// pairing whose grid it expects to finish first (lone_tile_first).
__host__ __device__ __forceinline__ int pair_first_tile(int n_qtiles, int lone_first, int pq) {
  if (!(n_qtiles & 1) || !lone_first) return 2 * pq;
  return pq == 0 ? 0 : 2 * pq - 1;
}
__host__ __device__ __forceinline__ bool pair_has_b(int n_qtiles, int lone_first, int pq) {
  if (!(n_qtiles & 1)) return true;
  return lone_first ? pq > 0 : 2 * pq + 1 < n_qtiles;
}

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
    w.q0[0] = pair_first_tile(p.n_qtiles, p.lone_first, pq) * BM;
    w.q0[1] = w.q0[0] + BM;
    w.has[0] = true;
    w.has[1] = pair_has_b(p.n_qtiles, p.lone_first, pq);
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

__device__ __forceinline__ void give_up_wait(volatile uint32_t* abort_flag, uint32_t code) {
  *abort_flag = 1u;
  const uint32_t cta = blockIdx.x < 0xFFFFFFu ? blockIdx.x : 0xFFFFFFu;
  atomicCAS(&g_fa_status, 0u, (code & 0xFFu) | (cta << 8));
}

// Slow path of a bounded wait: poll, then give up after the watchdog limit
// (or as soon as another role of this CTA has given up).  try_wait suspends
// until the phase completes or a hardware time limit, so the clock is read
// once per 32 polls; under a limit below 1 ms (a test making waits run out)
// it is read after every poll.  Two codings of that test path, chosen per
// kernel by measurement (the code around the normal loop changes how the
// kernels around it compile): kSeparate, a loop of its own (the two-tile and
// stream-K kernels), or an early exit from the normal loop (the hd 256 kernel).
template <bool kSeparate = true>
__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          unsigned long long limit_ns, uint32_t code) {
  const uint64_t t0 = ptx::globaltimer_ns();
  const bool fine = limit_ns < 1000000ull;
  if (kSeparate && fine) {
    while (!ptx::mbar_try_wait(bar, parity)) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > limit_ns) {
        give_up_wait(abort_flag, code);
        return false;
      }
    }
    return true;
  }
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i) {
      if (ptx::mbar_try_wait(bar, parity)) return true;
      if (!kSeparate && fine) break;
    }
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > limit_ns) {
      give_up_wait(abort_flag, code);
      return false;
    }
  }
}

template <bool kSeparate = true>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         unsigned long long limit_ns, uint32_t code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  return wait_slow<kSeparate>(bar, parity, abort_flag, limit_ns, code);
}

// Warp-uniform bounded wait (all 32 lanes call it; all get the same answer).
template <bool kSeparate = true>
__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity,
                                              volatile uint32_t* abort_flag,
                                              unsigned long long limit_ns, uint32_t code) {
  const bool ok = wait_bar<kSeparate>(bar, parity, abort_flag, limit_ns, code);
  return __all_sync(0xffffffffu, ok);
}

// The MMA warp's wait: warp-uniform when the whole warp runs the issue loop,
// else the single issuing thread's.
template <bool kWarp>
__device__ __forceinline__ bool mma_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         unsigned long long limit_ns, uint32_t code) {
  if constexpr (kWarp) return warp_wait_bar(bar, parity, abort_flag, limit_ns, code);
  else return wait_bar(bar, parity, abort_flag, limit_ns, code);
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
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                      const __grid_constant__ CUtensorMap tmKt, const __grid_constant__ CUtensorMap tmVt,
                      const Params p) {
  // heads up to 64 wide run on fa_prefill64_kernel (S and P apart in TMEM)
  static_assert(HD == 128, "the two-tile kernel with P over S is the 128-column one");
  using L = Layout<HD>;
  constexpr int NSLOT = L::NSLOT;
  // K/V arrive in pairs (V_j, K_j+1) on one barrier, so the MMA thread waits
  // once per KV step; K_0 arrives with Q.  Pair j+NPB reuses pair j's
  // barrier.  The producer arms it only once pair j has completed, and with
  // 2 NPB >= NSLOT it cannot complete before the MMA thread has waited for
  // pair j: its V's ring slot is freed only by P V(j) or a later MMA.
  constexpr int NPB = (NSLOT + 1) / 2;
  static_assert(2 * NPB >= NSLOT && NPB <= NSLOT, "pair barriers");
  // At hd 128, K_j and V_j free their ring slots together, on one commit
  // after P V_B(j) (one commit per step fewer for the MMA thread; measured
  // +0.5 to +0.8 %, and -2 % at hd 64, whose ring keeps per-slot frees).  The
  // producer waits on the pair-empty barrier of the slot's previous occupant;
  // with 2 NPE > NSLOT, pair j+NPE cannot be freed before the producer's waits
  // on pair j (its V is loaded only after them).
  constexpr bool PAIR_EMPTY = HD == 128;
  constexpr int NPE = NSLOT / 2 + 1;
  static_assert(2 * NPE > NSLOT && NPE <= NSLOT, "pair-empty barriers");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);

  const uint32_t sQ = sbase + L::OFF_Q;
  const uint32_t sRing = sbase + L::OFF_RING;
  const uint32_t bar = sbase + L::OFF_BAR;
  const uint32_t bQ = bar;
  auto bPair = [&](int b) { return bar + 8u * (1 + b); };  // b < NPB
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
    for (int b = 0; b < NPB; ++b) ptx::mbar_init(bPair(b), 2);  // one arrival per load of the pair
    for (int s = 0; s < NSLOT; ++s) ptx::mbar_init(bEmpty(s), 1);
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(bSfull(x), 1);
      ptx::mbar_init(bPfull(x), BM);  // one arrival per softmax thread of tile x
    }
    ptx::mbar_init(bOfinal, 1);
    ptx::mbar_init(bDrain, 1);
    misc[1] = 0u;
    // tile A's early o_final (row pairs, hd 128): the slot-free barrier of step nA-1
    uint32_t early_bar = 0u, early_par = 0u;
    if (HD == 128 && !p.pair_heads && nA > 0 && nA < n) {
      const int e = nA - 1;
      if constexpr (PAIR_EMPTY) {
        early_bar = bEmpty(e % NPE);
        early_par = (e / NPE) & 1;
      } else {
        early_bar = bEmpty((2 * e + 1) % NSLOT);
        early_par = ((2 * e + 1) / NSLOT) & 1;
      }
    }
    misc[2] = early_bar;
    misc[3] = early_par;
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
  // the set-up above overlaps the previous kernel's tail; nothing in global
  // memory is read or written before that kernel has completed
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();

  if (warp >= MMA_WARP) {
  ptx::setmaxnreg_dec<REGS_CONTROL>();
  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      ptx::prefetch_tmap(&tmO);
      ptx::mbar_arrive_expect_tx(bQ, L::Q_BYTES * (w.has[1] ? 2u : 1u) + (n > 0 ? L::SLOT_BYTES : 0u));
      for (int x = 0; x < 2; ++x) {
        if (!w.has[x]) continue;
#pragma unroll
        for (int c = 0; c < (int)L::KCH; ++c)
          ptx::tma_load_4d(sQ + x * L::Q_BYTES + c * (BM * 128), &tmQ, bQ, c * 64, w.hq[x], w.q0[x], w.b);
      }
      // loads in order K_0, V_0, K_1, V_1, ...; load i goes to slot i % NSLOT
      // (K_0 on bQ, then V_j and K_j+1 on pair barrier j % NPB)
      int issued = 0;
      bool ok = true;
      int page = -1, blk = 0;  // paged K/V: the pool block of the current page
      if (p.block_table) {
        ptx::prefetch_tmap(&tmKt);
        ptx::prefetch_tmap(&tmVt);
      }
      for (int i = 0; i < 2 * n; ++i) {
        const int s = i % NSLOT;
        if (i >= NSLOT) {
          if constexpr (PAIR_EMPTY) {  // the previous occupant, load i - NSLOT, belongs to pair e
            const int e = (i - NSLOT) >> 1;
            ok = wait_bar(bEmpty(e % NPE), (e / NPE) & 1, abort_flag, p.watchdog_ns, WD_PRODUCER_EMPTY);
          } else {
            ok = wait_bar(bEmpty(s), ((i / NSLOT) & 1) ^ 1u, abort_flag, p.watchdog_ns, WD_PRODUCER_EMPTY);
          }
        }
        if (!ok) break;
        const int key0 = (i >> 1) * BN;
        int row = key0, bat = w.b;
        bool tail = false;
        if (p.block_table) {
          const int pg = key0 / p.page_size;
          if (pg != page) {
            page = pg;
            blk = __ldg(p.block_table + static_cast<size_t>(w.b) * p.max_pages + pg);
            if (blk < 0 || blk >= p.num_blocks) {  // outside the pool: reported, and read one block
              atomicCAS(&g_fa_status, 0u,   // past the end, where TMA fills zeros
                        WD_PAGE_BLOCK | ((blockIdx.x < 0xFFFFFFu ? blockIdx.x : 0xFFFFFFu) << 8));
              blk = p.num_blocks;
            }
          }
          row = key0 - pg * p.page_size;
          bat = blk;
          tail = pg == p.last_page;
        }
        const int pj = (i - 1) >> 1;  // pair of load i (V_pj, K_pj+1)
        const uint32_t fb = i == 0 ? bQ : bPair(pj % NPB);
        // pair pj reuses pair pj-NPB's barrier: that phase must have completed
        if ((i & 1) && pj >= NPB) ok = wait_bar(fb, ((pj - NPB) / NPB) & 1, abort_flag, p.watchdog_ns, WD_PRODUCER_EMPTY);
        if (!ok) break;
        if (i > 0) ptx::mbar_arrive_expect_tx(fb, L::SLOT_BYTES);
        const CUtensorMap* m = (i & 1) ? (tail ? &tmVt : &tmV) : (tail ? &tmKt : &tmK);
#pragma unroll
        for (int c = 0; c < (int)L::KCH; ++c)
          ptx::tma_load_4d(sRing + s * L::SLOT_BYTES + c * (BN * 128), m, fb, c * 64, w.hk, row, bat);
        ++issued;
      }
      // a pair whose K was not issued (the last V, or a CTA that gave up):
      // its second arrival without bytes
      if (issued >= 2 && (issued & 1) == 0) ptx::mbar_arrive(bPair(((issued - 2) >> 1) % NPB));
      // every copy issued has landed before the CTA exits: in a normal run
      // the MMA thread consumed them all (these waits return at once); in a
      // CTA that gave up, some may still be in flight
      drain_wait(bQ, 0, DRAIN_NS);
      const int npairs = issued / 2;  // pairs armed
      for (int b = 0; b < NPB && b < npairs; ++b) {
        const int last = b + NPB * ((npairs - 1 - b) / NPB);
        drain_wait(bPair(b), (last / NPB) & 1, DRAIN_NS);
      }
    }
  } else if (warp == MMA_WARP) {
    // ----------------------------------------------------------- MMA issuer
    // lane 0 alone (a converged warp with one elected lane issuing measured
    // -5 to +2 % here; the hd 64 kernel, where it measured +6 %, uses it)
    if (lane == 0) {
      constexpr uint32_t IDESC_S = ptx::idesc_f16(BF16, BM, BN, false, false);  // Q, K both K-major
      constexpr uint32_t IDESC_O = ptx::idesc_f16(BF16, BM, HD, false, true);   // P from TMEM, V MN-major
      constexpr uint32_t DHI = ptx::sdesc_sw128_hi(1024);  // Q, K (K-major) and V (MN-major): SBO 1024
      auto issue_s = [&](int x, int slot) {
        const uint32_t d = tmem + L::TM_S + x * BN;
        const uint32_t q = ptx::sdesc_sw128_lo(sQ + x * L::Q_BYTES, 16);
        const uint32_t k = ptx::sdesc_sw128_lo(sRing + slot * L::SLOT_BYTES, 16);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t o = ((kk / 4) * (BM * 128) + (kk % 4) * 32) >> 4;
          ptx::mma_f16_ss(d, ptx::sdesc_join(q + o, DHI), ptx::sdesc_join(k + o, DHI), IDESC_S, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(bSfull(x));
      };
      auto issue_pv = [&](int x, int slot, bool acc) {
        const uint32_t d = tmem + L::TM_O + x * HD;
        const uint32_t a = tmem + L::TM_S + x * BN;  // P_X, 2 elements per column
        const uint32_t v = ptx::sdesc_sw128_lo(sRing + slot * L::SLOT_BYTES, BN * 128);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          ptx::mma_f16_ts(d, a + kk * 8, ptx::sdesc_join(v + kk * ((16 * 128) >> 4), DHI), IDESC_O,
                          (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = wait_bar(bQ, 0, abort_flag, p.watchdog_ns, WD_MMA_Q);  // Q and K_0
      if (ok && n > 0) {
        ptx::tc_fence_after();
        if (nA > 0) issue_s(0, 0);
        if (nB > 0) issue_s(1, 0);
        if constexpr (!PAIR_EMPTY) ptx::mma_commit(bEmpty(0));
      }
      for (int j = 0; ok && j < n; ++j) {
        const int iv = 2 * j + 1, sv = iv % NSLOT;  // V_j
        const int ik = 2 * j + 2, sk = ik % NSLOT;  // K_{j+1}
        const bool more = j + 1 < n;
        ok = wait_bar(bPair(j % NPB), (j / NPB) & 1, abort_flag, p.watchdog_ns, WD_MMA_KV_FULL);  // V_j, K_{j+1}
        if (!ok) break;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const int nX = x == 0 ? nA : nB;
          if (j < nX) {
            ok = wait_bar(bPfull(x), j & 1, abort_flag, p.watchdog_ns, WD_MMA_P_FULL);
            if (!ok) break;
            ptx::tc_fence_after();
            issue_pv(x, sv, j > 0);
          }
          if (x == 1) {
            if constexpr (PAIR_EMPTY)
              ptx::mma_commit(bEmpty(j % NPE));  // K_j (its S MMAs came earlier) and V_j, once P V_B(j) is done
            else
              ptx::mma_commit(bEmpty(sv));  // V_j no longer needed once PV_B(j) is done
          }
          if (more && j + 1 < nX) issue_s(x, sk);
        }
        if (!ok) break;
        if constexpr (!PAIR_EMPTY) {
          if (more) ptx::mma_commit(bEmpty(sk));
        }
      }
      if (ok) ptx::mma_commit(bOfinal);
      // every MMA issued has finished before TMEM is freed (the softmax may
      // have given up without waiting for o_final)
      ptx::mma_commit(bDrain);
      drain_wait(bDrain, 0, DRAIN_NS);
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
    // Once o_final has completed, no MMA reads the ring any more.  Row pairs
    // (tile B one KV tile longer than tile A): tile A's O is final once the
    // ring slots of step nA-1 are freed, a commit the MMA thread issues after
    // P V_B(nA-1) anyway, so tile A's epilogue runs under tile B's last step
    // (measured +2 % at 2048 and 2659 tokens, +13 % on one 256-token head;
    // no instruction added to the MMA thread).  No later commit reaches that
    // barrier: its next one would be step nA-1+NPE (or, per slot, load
    // 2 nA - 1 + NSLOT), past the last.  (Waited whenever the CTA streams any
    // KV tile, even if this tile has none.)
    // (The barrier and phase come from shared memory, set up by thread 0, so
    // the softmax keeps no extra register live through its loop.)
    if (ok && n > 0) {
      const bool early = HD == 128 && x == 0 && misc[2] != 0u;  // hd 64: -2.5 % from the code alone
      ok = warp_wait_bar(early ? misc[2] : bOfinal, early ? misc[3] : 0u, abort_flag, p.watchdog_ns,
                         WD_SOFTMAX_O_DONE);
      if (ok) ptx::tc_fence_after();
    }
    if (ok && hasx) {
      if (p.lse && q0 + r < p.Sq) p.lse[(static_cast<size_t>(w.b) * p.Hq + hqx) * p.Sq + q0 + r] = row_lse(m_ref, l);
      // O / l rounded to 16 bits, written 128-byte swizzled (the layout of a Q
      // tile) and sent out by TMA tensor stores, one per warp and 64-column
      // block: the global writes are whole lines, and rows past Sq are
      // clipped by the map.
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      // Stage slots: tile A in the slot of load 2n-4 (K_n-2), tile B in that
      // of load 2n-3 (V_n-2).  When tile A's O is final, only loads from
      // 2n-3 on can still be read (P V_B(n-2), S_B(n-1), P V_B(n-1)), and
      // no load is issued after 2n-1, so both slots stay free.
      const int stage_slot = (2 * n + 2 * NSLOT - 4 + x) % NSLOT;
      const uint32_t stage = sRing + stage_slot * L::SLOT_BYTES + r * 128;
      uint32_t orr[HD];  // the whole row: all loads in flight before one wait
      if (nX > 0) {
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) ptx::tmem_ld32(tO + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&orr[c * 32]));
        ptx::tmem_wait_ld();
        ptx::reg_fence(orr);
      } else {
#pragma unroll
        for (int e = 0; e < HD; ++e) orr[e] = 0u;
      }
#pragma unroll
      for (int ch = 0; ch < HD / 8; ++ch) {  // 16-byte chunk of the row: columns 8 ch .. 8 ch + 7
        const uint32_t* v = &orr[8 * ch];
        ptx::st_shared_v4(stage + (ch / 8) * (BM * 128) + (((ch % 8) ^ (r % 8)) * 16),
                          pack2<BF16>(__uint_as_float(v[0]) * inv_l, __uint_as_float(v[1]) * inv_l),
                          pack2<BF16>(__uint_as_float(v[2]) * inv_l, __uint_as_float(v[3]) * inv_l),
                          pack2<BF16>(__uint_as_float(v[4]) * inv_l, __uint_as_float(v[5]) * inv_l),
                          pack2<BF16>(__uint_as_float(v[6]) * inv_l, __uint_as_float(v[7]) * inv_l));
      }
      ptx::fence_proxy_async_smem();  // make the generic-proxy writes visible to the TMA unit
      __syncwarp();
      // each warp sends its own 32 rows (the map's box is 64 columns x 32
      // rows), so no warp waits for the tile's other three
      const int r0 = 32 * (warp & 3);
      if (lane == 0 && q0 + r0 < p.Sq) {
#pragma unroll
        for (int c = 0; c < (int)L::KCH; ++c)
          ptx::tma_store_4d(&tmO, sRing + stage_slot * L::SLOT_BYTES + c * (BM * 128) + r0 * 128, c * 64, hqx,
                            q0 + r0, w.b);
        ptx::bulk_commit();
        ptx::bulk_wait_read0();  // the slot must stay valid until the TMA unit has read it
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

}  // namespace fa

#include "fa_prefill256.cuh"
#include "fa_prefill64.cuh"
#include "fa_prefill_pair.cuh"

namespace fa {

// ================================================ stream-K (split-KV) kernel
//
// The one-shot kernel above gives every CTA whole query-tile pairs, so a grid
// with few pairs (a short chunk over a long context, one head) leaves SMs
// idle.  With no more pairs than SMs, the split-KV schedule cuts each pair
// into near-equal pieces of its KV steps, one per CTA, and this kernel runs
// them: every CTA computes one segment (unit u, KV steps [jb, je)) with the
// one-shot kernel's single step loop.  (Schedules with more pairs than SMs,
// where a CTA runs several segments, go to the persistent kernel in
// fa_persistent.cuh.)  A split pair's pieces each leave their unnormalised O,
// running max m and sum l in a workspace slot the host assigned, and a
// second, short kernel (fa_sk_merge_kernel, chained by programmatic dependent
// launch) combines them over the whole GPU in a fixed order, so results are
// deterministic.  No CTA waits on another.

constexpr int SK_MAX_CTAS = 256;
// The segment loop keeps more state in the control warps than the one-shot
// kernel: its own register split (same launch allocation).
constexpr uint32_t SK_REGS_SOFTMAX = 200;
constexpr uint32_t SK_REGS_CONTROL = 88;
static_assert(128 * SK_REGS_CONTROL + 256 * SK_REGS_SOFTMAX <= NUM_THREADS * LAUNCH_REGS,
              "register split exceeds the launch allocation");

// Workspace slots of split pieces: a CTA holds at most two (the tail of the
// pair its range starts in, the head of the pair its range ends in).
constexpr int SK_SLOTS = 2 * SK_MAX_CTAS;

struct SkParams {
  Params p;
  float4* ws_o;  // partial O, float4 [piece slot][tile][HD/4][BM]
  float* ws_ml;  // [piece slot][tile][2][BM]: m (log2 domain), l
  int su[SK_MAX_CTAS + 1];  // CTA c starts at pair unit su[c], KV step sj[c]; it ends where CTA c+1 starts
  int sj[SK_MAX_CTAS + 1];
  short pf[SK_MAX_CTAS];  // slot of CTA c's first segment when it continues a split pair, else -1
  short ph[SK_MAX_CTAS];  // slot of CTA c's last segment when it starts a split pair, else -1
};

template <int HD>
struct SkLayout {
  using L = Layout<HD>;
  // A persistent CTA keeps loading the next segment's K/V while it writes the
  // previous segment's O, so O cannot be staged in the ring: each softmax
  // thread writes its row straight from registers (or its piece to the
  // workspace), and the ring keeps the one-shot kernel's depth.
  static constexpr int NSLOT = HD == 128 ? 5 : 8;
  // q_full, full[NSLOT] (pair barriers: the first NPB), empty[NSLOT], s_full[2], p_full[2],
  // o_final[2], drain
  static constexpr uint32_t NUM_BARS = 1 + 2 * NSLOT + 2 + 2 + 2 + 1;
  static constexpr uint32_t OFF_BAR = L::OFF_RING + NSLOT * L::SLOT_BYTES;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static constexpr uint32_t REQUEST = BYTES + 1024;
  static constexpr size_t WS_O_BYTES = (size_t)SK_SLOTS * 2 * BM * HD * 4;
  static constexpr size_t WS_ML_BYTES = (size_t)SK_SLOTS * 2 * 2 * BM * 4;
  static constexpr size_t WS_BYTES = WS_O_BYTES + WS_ML_BYTES;
};

// Geometry of pair unit u (same numbering as the one-shot grid: longest
// first; G/2 pairs of one KV group adjacent).  Host and device share it so the
// host's schedule and the kernel's decode cannot disagree.
struct UnitGeo {
  int b, hk, hq0, hq1, q00, q01;
  bool has1;
  int nA, nB, n;
};

__host__ __device__ __forceinline__ int geo_kv_tiles(const Params& p, int q0) {
  const int off = p.Skv - p.Sq;
  const int q_last = (q0 + BM < p.Sq ? q0 + BM : p.Sq) - 1;
  int kv_hi = p.Skv;
  if (p.causal) kv_hi = (off + q_last + 1 < p.Skv) ? off + q_last + 1 : p.Skv;
  return kv_hi > 0 ? (kv_hi + BN - 1) / BN : 0;
}

__host__ __device__ __forceinline__ UnitGeo unit_geo(const Params& p, int u) {
  UnitGeo w;
  if (p.pair_heads) {
    const int pairs = p.Hq / 2;
    const int per_qt = pairs * p.B;
    const int qt = p.n_qtiles - 1 - u / per_qt;
    const int rem = u % per_qt;
    w.b = rem / pairs;
    const int pi = rem % pairs;
    w.hq0 = 2 * pi;
    w.hq1 = 2 * pi + 1;
    w.q00 = w.q01 = qt * BM;
    w.has1 = true;
  } else {
    const int npq = (p.n_qtiles + 1) / 2;
    const int per = p.Hq * p.B;
    const int pq = npq - 1 - u / per;
    const int rem = u % per;
    w.b = rem / p.Hq;
    w.hq0 = w.hq1 = rem % p.Hq;
    w.q00 = pair_first_tile(p.n_qtiles, p.lone_first, pq) * BM;
    w.q01 = w.q00 + BM;
    w.has1 = pair_has_b(p.n_qtiles, p.lone_first, pq);
  }
  w.hk = w.hq0 / p.G;
  w.nA = geo_kv_tiles(p, w.q00);
  w.nB = w.has1 ? geo_kv_tiles(p, w.q01) : 0;
  w.n = w.nA > w.nB ? w.nA : w.nB;
  return w;
}

template <int HD, bool BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fa_prefill_sk_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                         const __grid_constant__ CUtensorMap tmKt, const __grid_constant__ CUtensorMap tmVt,
                         const __grid_constant__ SkParams sp) {
  const Params& p = sp.p;
  using L = Layout<HD>;
  using SL = SkLayout<HD>;
  constexpr int NSLOT = SL::NSLOT;
  // One-segment CTAs take the one-shot kernel's K/V protocol: K_jb arrives
  // with Q, then V_t and K_t+1 on pair barrier t % NPB (full[0 .. NPB)), one
  // wait per step for the MMA thread (same reuse rule: 2 NPB >= NSLOT).
  constexpr int NPB = (NSLOT + 1) / 2;
  static_assert(2 * NPB >= NSLOT && NPB <= NSLOT, "pair barriers");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);

  const uint32_t sQ = sbase + L::OFF_Q;
  const uint32_t sRing = sbase + L::OFF_RING;
  const uint32_t bar = sbase + SL::OFF_BAR;
  const uint32_t bQfull = bar;
  auto bFull = [&](int s) { return bar + 8u * (1 + s); };
  auto bEmpty = [&](int s) { return bar + 8u * (1 + NSLOT + s); };
  auto bSfull = [&](int x) { return bar + 8u * (1 + 2 * NSLOT + x); };
  auto bPfull = [&](int x) { return bar + 8u * (3 + 2 * NSLOT + x); };
  auto bOfinal = [&](int x) { return bar + 8u * (5 + 2 * NSLOT + x); };
  const uint32_t bDrain = bar + 8u * (7 + 2 * NSLOT);
  uint32_t* misc = reinterpret_cast<uint32_t*>(gbase + SL::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = static_cast<int>(blockIdx.x);
  // this CTA's one segment: unit u, KV steps [jb, je) (it ends where the next
  // CTA starts, or at the unit's end)
  const int u = sp.su[cta], jb = sp.sj[cta];
  const UnitGeo w = unit_geo(p, u);
  const int je = (sp.su[cta + 1] == u) ? sp.sj[cta + 1] : w.n;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bQfull, 1);
    for (int s = 0; s < NSLOT; ++s) {
      ptx::mbar_init(bFull(s), s < NPB ? 2 : 1);  // pair barriers (the first NPB): one arrival per load
      ptx::mbar_init(bEmpty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(bSfull(x), 1);
      ptx::mbar_init(bPfull(x), BM);  // one arrival per softmax thread of tile x
      ptx::mbar_init(bOfinal(x), 1);
    }
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
  // as in the one-shot kernel: set-up overlaps the previous kernel; no global
  // access before it has completed.  The merge kernel may launch early too.
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();

  if (warp >= MMA_WARP) {
    ptx::setmaxnreg_dec<SK_REGS_CONTROL>();
    if (warp == PRODUCER_WARP && lane == 0) {
      // ---------------------------------------------------------- producer
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      ptx::prefetch_tmap(&tmO);
      if (p.block_table) {
        ptx::prefetch_tmap(&tmKt);
        ptx::prefetch_tmap(&tmVt);
      }
      int g = 0;  // loads issued into the ring: K_jb, then pairs (V_t, K_t+1)
      bool ok = true;
      if (je > jb) {  // else nothing to stream (the softmax writes zeros)
        ptx::mbar_arrive_expect_tx(bQfull, L::Q_BYTES * (w.has1 ? 2u : 1u) + L::SLOT_BYTES);
#pragma unroll
        for (int c = 0; c < (int)L::KCH; ++c)
          ptx::tma_load_4d(sQ + c * (BM * 128), &tmQ, bQfull, c * 64, w.hq0, w.q00, w.b);
        if (w.has1) {
#pragma unroll
          for (int c = 0; c < (int)L::KCH; ++c)
            ptx::tma_load_4d(sQ + L::Q_BYTES + c * (BM * 128), &tmQ, bQfull, c * 64, w.hq1, w.q01, w.b);
        }
        int page = -1, blk = 0;  // paged K/V: the pool block of the current page
        for (int i = 2 * jb; i < 2 * je; ++i, ++g) {
          const int s = g % NSLOT;
          if (g >= NSLOT) ok = wait_bar(bEmpty(s), ((g / NSLOT) & 1) ^ 1u, abort_flag, p.watchdog_ns, WD_PRODUCER_EMPTY);
          if (!ok) break;
          const int key0 = (i >> 1) * BN;
          int row = key0, bat = w.b;
          bool tail = false;
          if (p.block_table) {  // as in the one-shot producer
            const int pg = key0 / p.page_size;
            if (pg != page) {
              page = pg;
              blk = __ldg(p.block_table + static_cast<size_t>(w.b) * p.max_pages + pg);
              if (blk < 0 || blk >= p.num_blocks) {
                atomicCAS(&g_fa_status, 0u,
                          WD_PAGE_BLOCK | ((blockIdx.x < 0xFFFFFFu ? blockIdx.x : 0xFFFFFFu) << 8));
                blk = p.num_blocks;
              }
            }
            row = key0 - pg * p.page_size;
            bat = blk;
            tail = pg == p.last_page;
          }
          const int pj = (g - 1) >> 1;  // pair of load g (V_pj, K_pj+1); K_jb comes with Q
          const uint32_t fb = g == 0 ? bQfull : bFull(pj % NPB);
          if ((g & 1) && pj >= NPB) {  // pair pj reuses pair pj-NPB's barrier
            ok = wait_bar(fb, ((pj - NPB) / NPB) & 1, abort_flag, p.watchdog_ns, WD_PRODUCER_EMPTY);
            if (!ok) break;
          }
          if (g > 0) ptx::mbar_arrive_expect_tx(fb, L::SLOT_BYTES);
          const CUtensorMap* m = (i & 1) ? (tail ? &tmVt : &tmV) : (tail ? &tmKt : &tmK);
#pragma unroll
          for (int c = 0; c < (int)L::KCH; ++c)
            ptx::tma_load_4d(sRing + s * L::SLOT_BYTES + c * (BN * 128), m, fb, c * 64, w.hk, row, bat);
        }
      }
      // a pair whose K was not issued (the last V, or a CTA that gave up)
      if (g >= 2 && (g & 1) == 0) ptx::mbar_arrive(bFull(((g - 2) >> 1) % NPB));
      // every copy issued has landed before the CTA exits (as in the one-shot kernel)
      if (je > jb) drain_wait(bQfull, 0, DRAIN_NS);
      const int npairs = g / 2;  // pairs armed
      for (int b = 0; b < NPB && b < npairs; ++b) {
        const int last = b + NPB * ((npairs - 1 - b) / NPB);
        drain_wait(bFull(b), (last / NPB) & 1, DRAIN_NS);
      }
    } else if (warp == MMA_WARP && lane == 0) {
      // ------------------------------------------------------- MMA issuer
      constexpr uint32_t IDESC_S = ptx::idesc_f16(BF16, BM, BN, false, false);
      constexpr uint32_t IDESC_O = ptx::idesc_f16(BF16, BM, HD, false, true);
      constexpr uint32_t DHI = ptx::sdesc_sw128_hi(1024);  // Q, K (K-major) and V (MN-major): SBO 1024
      auto issue_s = [&](int x, int slot) {
        const uint32_t d = tmem + L::TM_S + x * BN;
        const uint32_t q = ptx::sdesc_sw128_lo(sQ + x * L::Q_BYTES, 16);
        const uint32_t k = ptx::sdesc_sw128_lo(sRing + slot * L::SLOT_BYTES, 16);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t o = ((kk / 4) * (BM * 128) + (kk % 4) * 32) >> 4;
          ptx::mma_f16_ss(d, ptx::sdesc_join(q + o, DHI), ptx::sdesc_join(k + o, DHI), IDESC_S, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(bSfull(x));
      };
      auto issue_pv = [&](int x, int slot, bool acc) {
        const uint32_t d = tmem + L::TM_O + x * HD;
        const uint32_t a = tmem + L::TM_S + x * BN;
        const uint32_t v = ptx::sdesc_sw128_lo(sRing + slot * L::SLOT_BYTES, BN * 128);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          ptx::mma_f16_ts(d, a + kk * 8, ptx::sdesc_join(v + kk * ((16 * 128) >> 4), DHI), IDESC_O,
                          (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = true;
      if (je > jb) {
        const int nseg = je - jb;
        const int nAs = max(0, min(je, w.nA) - jb);  // tiles of A / B in this segment
        const int nBs = max(0, min(je, w.nB) - jb);
        ok = wait_bar(bQfull, 0, abort_flag, p.watchdog_ns, WD_MMA_Q);  // Q and K_jb
        if (ok) {
          ptx::tc_fence_after();
          if (nAs > 0) issue_s(0, 0);
          if (nBs > 0) issue_s(1, 0);
          ptx::mma_commit(bEmpty(0));
        }
        // ring index of V_(jb+t) is 2t + 1, of K_(jb+t+1) 2t + 2; both on pair barrier t % NPB
        for (int t = 0; ok && t < nseg; ++t) {
          const int sv = (2 * t + 1) % NSLOT;
          const int sk = (2 * t + 2) % NSLOT;
          const bool more = t + 1 < nseg;
          ok = wait_bar(bFull(t % NPB), (t / NPB) & 1, abort_flag, p.watchdog_ns, WD_MMA_KV_FULL);  // V_t, K_t+1
          if (!ok) break;
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            const int nXs = x == 0 ? nAs : nBs;
            if (t < nXs) {
              ok = wait_bar(bPfull(x), t & 1, abort_flag, p.watchdog_ns, WD_MMA_P_FULL);
              if (!ok) break;
              ptx::tc_fence_after();
              issue_pv(x, sv, t > 0);
            }
            if (x == 1) ptx::mma_commit(bEmpty(sv));
            if (more && t + 1 < nXs) issue_s(x, sk);
          }
          if (!ok) break;
          if (more) ptx::mma_commit(bEmpty(sk));
        }
        if (ok && nAs > 0) ptx::mma_commit(bOfinal(0));
        if (ok && nBs > 0) ptx::mma_commit(bOfinal(1));
      }
      // every MMA issued has finished before TMEM is freed
      ptx::mma_commit(bDrain);
      drain_wait(bDrain, 0, DRAIN_NS);
    }
  } else {
    ptx::setmaxnreg_inc<SK_REGS_SOFTMAX>();
    // -------------------------------------------------------------- softmax
    const int x = warp >> 2;
    const int r = threadIdx.x & 127;
    const int wq = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + L::TM_S + x * BN;
    const uint32_t tO = tmem + lane_off + L::TM_O + x * HD;
    const int off = p.Skv - p.Sq;
    const float sl2 = p.sl2;
    int cnt = 0;   // tiles processed (s_full / p_full phases)
    int ocnt = 0;  // segments with tiles of x (o_final phases)
    bool ok = true;
    do {
      const bool first = jb == 0;
      const bool last = je >= w.n;
      const int q0 = x == 0 ? w.q00 : w.q01;
      const int hqx = x == 0 ? w.hq0 : w.hq1;
      const bool hasx = x == 0 ? true : w.has1;
      const int nX = x == 0 ? w.nA : w.nB;
      const int jx_end = min(je, nX);
      const int ntile = max(0, jx_end - jb);
      const int kv_all = p.causal ? min(p.Skv, off + q0 + 1) : p.Skv;
      const int row_lim = p.causal ? min(p.Skv, off + q0 + r + 1) : p.Skv;
      float m_ref = -INFINITY;
      float l = 0.f;
      for (int j = jb; j < jx_end; ++j, ++cnt) {
        ok = warp_wait_bar(bSfull(x), cnt & 1, abort_flag, p.watchdog_ns, WD_SOFTMAX_S_FULL);
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t sr[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
          ptx::tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
        ptx::tmem_wait_ld();
        ptx::reg_fence(sr);
        float s[BN];
#pragma unroll
        for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(sr[c]);
        const int kv0 = j * BN;
        if (kv0 + BN > kv_all) {
          const int lim = row_lim - kv0;
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c >= lim) s[c] = -INFINITY;
        }
        float mk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mk[k] = ptx::fmax3(s[k], s[8 + k], s[16 + k]);
#pragma unroll
        for (int t = 3; t < 15; t += 2)
#pragma unroll
          for (int k = 0; k < 8; ++k) mk[k] = ptx::fmax3(mk[k], s[8 * t + k], s[8 * t + 8 + k]);
#pragma unroll
        for (int k = 0; k < 8; ++k) mk[k] = fmaxf(mk[k], s[120 + k]);
        const float mx =
            ptx::fmax3(ptx::fmax3(mk[0], mk[1], mk[2]), ptx::fmax3(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7]));
        const float m_new = fmaxf(m_ref, mx * sl2);
        const bool resc = m_new > m_ref + RESCALE_TAU;
        float alpha = 1.f;
        if (resc) {
          alpha = ptx::ex2(m_ref - m_new);
          m_ref = m_new;
          l *= alpha;
        }
        const float mb = (m_ref == -INFINITY) ? 0.f : m_ref;
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
        if (j > jb && __any_sync(0xffffffffu, resc)) {
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
        ptx::tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pp[0]));
        ptx::tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pp[32]));
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bPfull(x));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (ntile > 0) {
        ok = warp_wait_bar(bOfinal(x), ocnt & 1, abort_flag, p.watchdog_ns, WD_SOFTMAX_O_DONE);
        if (!ok) break;
        ++ocnt;
        ptx::tc_fence_after();
      }
      if (!hasx) continue;
      if (!(first && last)) {
        // a piece of a split pair: (O, m, l) to its slot; the merge kernel
        // writes the pair's output
        const int ps = first ? sp.ph[cta] : sp.pf[cta];
        if (ps < 0) {
          const uint32_t ci = blockIdx.x < 0xFFFFFFu ? blockIdx.x : 0xFFFFFFu;
          atomicCAS(&g_fa_status, 0u, WD_PIECE_SLOT | (ci << 8));
          continue;
        }
        const size_t slot_t = static_cast<size_t>(ps) * 2 + x;
        if (ntile > 0) {
          float4* dst = sp.ws_o + slot_t * (HD / 4) * BM + r;
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t orr[32];
            ptx::tmem_ld32(tO + c * 32, orr);
            ptx::tmem_wait_ld();
            ptx::reg_fence(orr);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[(c * 8 + e) * BM] = make_float4(__uint_as_float(orr[4 * e]), __uint_as_float(orr[4 * e + 1]),
                                                  __uint_as_float(orr[4 * e + 2]), __uint_as_float(orr[4 * e + 3]));
          }
        }
        sp.ws_ml[(slot_t * 2 + 0) * BM + r] = ntile > 0 ? m_ref : -INFINITY;
        sp.ws_ml[(slot_t * 2 + 1) * BM + r] = ntile > 0 ? l : 0.f;
        continue;
      }
      // a whole pair: O / l straight out
      const float M = ntile > 0 ? m_ref : -INFINITY;
      const float Lsum = ntile > 0 ? l : 0.f;
      const float inv_l = (Lsum > 0.f) ? 1.f / Lsum : 0.f;
      if (p.lse && q0 + r < p.Sq) p.lse[(static_cast<size_t>(w.b) * p.Hq + hqx) * p.Sq + q0 + r] = row_lse(M, Lsum);
      // O / l rounded to 16 bits, from registers straight to the row (the ring
      // is already filling with the next segment's K/V): whole 32-byte sectors
      // where the row is 32-byte aligned, up to the head's true width
      uint32_t orr[HD];
      if (ntile > 0) {
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) ptx::tmem_ld32(tO + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&orr[c * 32]));
        ptx::tmem_wait_ld();
        ptx::reg_fence(orr);
      } else {
#pragma unroll
        for (int e = 0; e < HD; ++e) orr[e] = 0u;
      }
      if (q0 + r < p.Sq) {
        uint16_t* orow = p.o + ((static_cast<size_t>(w.b) * p.Sq + q0 + r) * p.Hq + hqx) * p.hd;
        const bool a32 = (reinterpret_cast<uintptr_t>(orow) & 31u) == 0;
#pragma unroll
        for (int g = 0; g < HD / 16; ++g) {
          if (16 * g >= p.hd) break;
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            pk[e] = pack2<BF16>(__uint_as_float(orr[16 * g + 2 * e]) * inv_l, __uint_as_float(orr[16 * g + 2 * e + 1]) * inv_l);
          if (a32 && 16 * g + 16 <= p.hd) {
            ptx::st_global_v8(orow + 16 * g, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
          } else {
            *reinterpret_cast<uint4*>(orow + 16 * g) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            if (16 * g + 8 < p.hd) *reinterpret_cast<uint4*>(orow + 16 * g + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
    } while (false);  // one segment (a `continue` above ends it)
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ========================================================= split-pair merge
//
// After the stream-K kernel: one CTA per (split pair, query tile, 32-row
// block, 64-column half).  Each thread owns one row and eight output columns
// and combines the pair's pieces in slot order (the piece holding KV tile 0
// first, then the later pieces in CTA order), as online-softmax tiles combine:
// M = max m_k, O = sum 2^(m_k - M) O_k / sum 2^(m_k - M) l_k.  A piece that saw
// no key of a row (m = -inf) contributes nothing and its O is not read.
constexpr int MERGE_THREADS = 256;  // 8 warps: one 8-column chunk each, lanes = rows

struct MergeParams {
  Params p;
  const float4* ws_o;  // as SkParams
  const float* ws_ml;
  int n_split;
  int mu[SK_MAX_CTAS];    // split pair unit
  short ms[SK_MAX_CTAS];  // its first piece's slot; pieces at ms .. ms + mn - 1 in KV order
  short mn[SK_MAX_CTAS];
};

template <int HD, bool BF16>
__global__ void __launch_bounds__(MERGE_THREADS)
    fa_sk_merge_kernel(const __grid_constant__ MergeParams mp) {
  const Params& p = mp.p;
  constexpr int HALVES = HD / 64;  // 64-column halves (hd 128) or the whole row (hd 64)
  const int blk = static_cast<int>(blockIdx.x);
  const int hf = blk % HALVES;
  const int rb = (blk / HALVES) % (BM / 32);
  const int x = (blk / (HALVES * (BM / 32))) & 1;
  const int i = blk / (HALVES * (BM / 32) * 2);
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();  // every piece of the stream-K kernel is written and visible
  if (i >= mp.n_split) return;
  const UnitGeo w = unit_geo(p, mp.mu[i]);
  if (x == 1 && !w.has1) return;
  const int q0 = x == 0 ? w.q00 : w.q01;
  const int hq = x == 0 ? w.hq0 : w.hq1;
  const int lane = threadIdx.x & 31;
  const int r = rb * 32 + lane;
  const int ch = hf * 8 + (threadIdx.x >> 5);  // 8-column chunk: float4 groups 2 ch, 2 ch + 1
  const int s0 = mp.ms[i], np = mp.mn[i];
  auto ml = [&](int k, int which) { return mp.ws_ml[((static_cast<size_t>(s0 + k) * 2 + x) * 2 + which) * BM + r]; };
  float M = -INFINITY;
  for (int k = 0; k < np; ++k) M = fmaxf(M, ml(k, 0));
  float L = 0.f;
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int k = 0; k < np; ++k) {
    const float mk = ml(k, 0);
    const bool vk = mk != -INFINITY;
    const float f = vk ? ptx::ex2(mk - M) : 0.f;
    const float lk = ml(k, 1);
    const float4* src = mp.ws_o + (static_cast<size_t>(s0 + k) * 2 + x) * (HD / 4) * BM + r;
    float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
    if (vk) {
      v0 = src[(2 * ch) * BM];
      v1 = src[(2 * ch + 1) * BM];
    }
    L = vk ? fmaf(lk, f, L) : L;
    a[0] = vk ? fmaf(v0.x, f, a[0]) : a[0];
    a[1] = vk ? fmaf(v0.y, f, a[1]) : a[1];
    a[2] = vk ? fmaf(v0.z, f, a[2]) : a[2];
    a[3] = vk ? fmaf(v0.w, f, a[3]) : a[3];
    a[4] = vk ? fmaf(v1.x, f, a[4]) : a[4];
    a[5] = vk ? fmaf(v1.y, f, a[5]) : a[5];
    a[6] = vk ? fmaf(v1.z, f, a[6]) : a[6];
    a[7] = vk ? fmaf(v1.w, f, a[7]) : a[7];
  }
  if (q0 + r >= p.Sq) return;
  if (ch == 0 && p.lse) p.lse[(static_cast<size_t>(w.b) * p.Hq + hq) * p.Sq + q0 + r] = row_lse(M, L);
  if (8 * ch >= p.hd) return;  // zero padding columns of a narrower head
  const float inv = L > 0.f ? 1.f / L : 0.f;
  uint16_t* orow = p.o + ((static_cast<size_t>(w.b) * p.Sq + q0 + r) * p.Hq + hq) * p.hd + 8 * ch;
  *reinterpret_cast<uint4*>(orow) = make_uint4(pack2<BF16>(a[0] * inv, a[1] * inv), pack2<BF16>(a[2] * inv, a[3] * inv),
                                               pack2<BF16>(a[4] * inv, a[5] * inv), pack2<BF16>(a[6] * inv, a[7] * inv));
}

}  // namespace fa

#include "fa_persistent.cuh"

namespace fa {

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

// 4-D map over a BSHD tensor: dims (hd, H, S, B), box (64, 1, box_rows, 1), 128-byte swizzle.
// A [B][S_stride][H][hd] 16-bit tensor of which rows [0, S) of each batch are
// described: rows from S on are out of bounds for the map, so TMA loads them
// as zeros (S_stride = S for a contiguous BSHD tensor; a KV cache's capacity
// otherwise).
static bool encode_bshd(CUtensorMap* m, EncodeTiledFn enc, const void* base, bool bf16, int B, int S, int H, int hd,
                        int S_stride, int box_rows = 128) {
  const cuuint64_t rows = (cuuint64_t)(S > 0 ? S : 1), rows_mem = (cuuint64_t)(S_stride > S ? S_stride : rows);
  const cuuint64_t dims[4] = {(cuuint64_t)hd, (cuuint64_t)H, rows, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)hd * 2, (cuuint64_t)H * hd * 2, rows_mem * H * hd * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
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

// Pair units of a launch (the one-shot kernel's grid size).
static long long unit_count_of(const Params& p) {
  const long long n_qt = p.n_qtiles;
  if (p.pair_heads) return n_qt * (p.Hq / 2) * p.B;
  return ((n_qt + 1) / 2) * (long long)p.Hq * p.B;
}

// Row-pair grids with an odd tile count: which tile goes without a partner
// (pair_first_tile).  A list-scheduling model of the one-shot grid (CTAs in
// launch order, each to the SM that frees first) decides: a CTA costs its KV
// steps -- 0.65 of a step each when it holds one tile, whose chain leaves the
// tensor core idle much of the time -- plus 2.5 steps of fixed cost.  Tile 0
// alone cuts the grid's total steps, which counts from ~1.5 waves on (2432
// and 2659-token MHA prefills measured +6 % and +3 %, 24 heads of GQA 3
// +5.5 %); near one wave the longest CTA sets the time, and a pair there is
// slower than the last tile alone (1152 tokens: -8 %), as the model has it.
// Cached per shape.
static int lone_tile_first(const Params& prm0, int sms) {
  if (prm0.pair_heads || !(prm0.n_qtiles & 1) || prm0.n_qtiles < 3 || sms < 1) return 0;
  const long long nu = unit_count_of(prm0);
  if (nu > (1 << 16)) return 1;  // many waves: the total decides
  static std::mutex mu;
  static int cache[8][8];
  static int n_cached = 0, next = 0;
  const int key[7] = {prm0.B, prm0.Hq, prm0.Hkv, prm0.Sq, prm0.Skv, prm0.causal, sms};
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < n_cached; ++i)
      if (std::memcmp(cache[i], key, sizeof(key)) == 0) return cache[i][7];
  }
  double span[2];
  for (int lf = 0; lf < 2; ++lf) {
    Params prm = prm0;
    prm.lone_first = lf;
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    for (int i = 0; i < sms; ++i) free_at.push(0.0);
    span[lf] = 0.0;
    for (long long u = 0; u < nu; ++u) {
      const UnitGeo w = unit_geo(prm, static_cast<int>(u));
      const double t = free_at.top() + (w.has1 ? w.n : 0.65 * w.n) + 2.5;
      free_at.pop();
      free_at.push(t);
      span[lf] = std::max(span[lf], t);
    }
  }
  const int lf = span[1] < 0.99 * span[0] ? 1 : 0;
  std::lock_guard<std::mutex> lk(mu);
  std::memcpy(cache[next], key, sizeof(key));
  cache[next][7] = lf;
  next = (next + 1) % 8;
  if (n_cached < 8) ++n_cached;
  return lf;
}

constexpr int MAX_DEVICES = 64;

// The wait limit the next launches give their kernels (fa_debug_set_watchdog_ns).
static std::atomic<unsigned long long> g_watchdog_ns{WATCHDOG_NS};

// Per-device facts, filled once: 1 = sm_103 with enough opt-in shared memory.
static std::atomic<int> g_dev_ok[MAX_DEVICES];
static std::atomic<int> g_dev_sms[MAX_DEVICES];
static std::atomic<int> g_attr_set[MAX_DEVICES][4];
static std::atomic<int> g_sk_attr_set[MAX_DEVICES][8];
static std::atomic<int> g_pk_attr_set[MAX_DEVICES][4];
// Kernel selection for testing and measurement (fa_debug_force_path): 0 the
// library's choice, 1 the one-shot kernel (also for calls with a workspace),
// 2 the persistent kernel (over whole units without a workspace; for every
// split-KV schedule with one), 3 the CTA-pair kernel where it applies (GQA
// groups of a multiple of 4 query heads, heads 72 to 128 wide, contiguous
// K/V; measured slower than the single-CTA kernel, so never chosen by default).
static std::atomic<int> g_force_path{0};
static std::atomic<int> g_attr256_set[MAX_DEVICES][2];

static int check_device(int* dev_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
    (void)cudaGetLastError();
    return FA_ERR_DEVICE;
  }
  *dev_out = dev;
  int st = g_dev_ok[dev].load();
  if (st == 0) {
    int major = 0, minor = 0, optin = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      return FA_ERR_DEVICE;
    }
    g_dev_sms[dev].store(sms > 0 ? sms : 1);
    if (major != 10 || minor != 3) st = -FA_ERR_DEVICE;
    else if ((unsigned)optin < Layout<128>::REQUEST || (unsigned)optin < SkLayout<128>::REQUEST ||
             (unsigned)optin < Layout256::REQUEST || (unsigned)optin < PkLayout<128>::REQUEST ||
             (unsigned)optin < PairLayout::REQUEST)
      st = -FA_ERR_SMEM;
    else st = 1;
    g_dev_ok[dev].store(st);
  }
  return st == 1 ? FA_OK : -st;
}

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na > 0 && nb > 0 && x < y + nb && y < x + na;
}

// Launch with programmatic stream serialization: the kernel's set-up (barrier
// init, TMEM allocation) may overlap the previous kernel in the stream; the
// kernel waits (griddepcontrol.wait) before it reads or writes global memory,
// so it still sees everything the previous kernel wrote.
template <typename... P, typename... A>
static cudaError_t launch_pdl(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, A&&... args) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}

// Paged K/V: pool [num_blocks][page_size][Hkv][hd], block table [B][max_pages].
struct Paged {
  const int* table;
  int page_size, max_pages, num_blocks;
};

template <int HD, bool BF16>
static int launch_pk(const void* q, const void* k, const void* v, void* o, int hd, int B, int Hq, int Hkv, int Sq, int Skv,
                     int kv_cap, int causal, float scale, float4* ws_o, float* ws_ml, cudaStream_t stream, int dev,
                     const Paged* pg = nullptr, float* lse = nullptr);

// K/V maps for the producers, and the paged fields of Params.  Contiguous:
// Skv rows per sequence with a batch stride of kv_cap rows (the tail maps
// repeat the main ones).  Paged: whole pages through the pool maps, the last
// page through maps that end at its last valid row, so rows past Skv load as
// zeros.
static bool encode_kv(CUtensorMap* mk, CUtensorMap* mv, CUtensorMap* mkt, CUtensorMap* mvt, EncodeTiledFn enc,
                      const void* k, const void* v, bool bf16, int B, int Skv, int kv_cap, int Hkv, int hd,
                      const Paged* pg, Params* prm) {
  prm->block_table = nullptr;
  prm->page_size = prm->max_pages = prm->num_blocks = prm->last_page = 0;
  if (pg && Skv > 0) {
    const int last_page = (Skv - 1) / pg->page_size;
    const int tail_rows = Skv - last_page * pg->page_size;
    if (!encode_bshd(mk, enc, k, bf16, pg->num_blocks, pg->page_size, Hkv, hd, pg->page_size) ||
        !encode_bshd(mv, enc, v, bf16, pg->num_blocks, pg->page_size, Hkv, hd, pg->page_size) ||
        !encode_bshd(mkt, enc, k, bf16, pg->num_blocks, tail_rows, Hkv, hd, pg->page_size) ||
        !encode_bshd(mvt, enc, v, bf16, pg->num_blocks, tail_rows, Hkv, hd, pg->page_size))
      return false;
    prm->block_table = pg->table;
    prm->page_size = pg->page_size;
    prm->max_pages = pg->max_pages;
    prm->num_blocks = pg->num_blocks;
    prm->last_page = last_page;
    return true;
  }
  if (!encode_bshd(mk, enc, k, bf16, B, Skv, Hkv, hd, kv_cap) || !encode_bshd(mv, enc, v, bf16, B, Skv, Hkv, hd, kv_cap))
    return false;
  *mkt = *mk;
  *mvt = *mv;
  return true;
}

// The CTA-pair kernel (fa_prefill_pair.cuh): heads 72 to 128 wide, contiguous
// K/V, GQA groups of a multiple of 4 query heads.  Two CTAs per unit of four
// heads at one 128-row block.  Run only when asked for (fa_debug_force_path(3)):
// on the 8192-token GQA prefill it measured 504 us per call against 341 us
// for the single-CTA kernel.
static std::atomic<int> g_pair_attr_set[MAX_DEVICES][2];

static bool pair_applies(int Hq, int Hkv, const Paged* pg) {
  return g_force_path.load() == 3 && pg == nullptr && (Hq / Hkv) % 4 == 0;
}

template <bool BF16>
static int launch_pair(const void* q, const void* k, const void* v, void* o, int hd, int B, int Hq, int Hkv, int Sq,
                       int Skv, int kv_cap, int causal, float scale, cudaStream_t stream, int dev, float* lse) {
  auto kern = fa_prefill_pair_kernel<BF16>;
  const int slot = BF16 ? 1 : 0;
  if (g_pair_attr_set[dev][slot].load() == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PairLayout::REQUEST) !=
        cudaSuccess) {
      (void)cudaGetLastError();
      return FA_ERR_SMEM;
    }
    g_pair_attr_set[dev][slot].store(1);
  }
  EncodeTiledFn enc = encoder();
  if (!enc) return FA_ERR_LAUNCH;
  CUtensorMap mq, mkh, mv, mo;
  if (!encode_bshd(&mq, enc, q, BF16, B, Sq, Hq, hd, Sq) || !encode_bshd(&mo, enc, o, BF16, B, Sq, Hq, hd, Sq) ||
      !encode_bshd(&mkh, enc, k, BF16, B, Skv, Hkv, hd, kv_cap, 64) ||
      !encode_bshd(&mv, enc, v, BF16, B, Skv, Hkv, hd, kv_cap))
    return FA_ERR_LAUNCH;
  Params prm;
  std::memset(&prm, 0, sizeof(prm));
  prm.lse = lse;
  prm.o = static_cast<uint16_t*>(o);
  prm.hd = hd;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Sq = Sq;
  prm.Skv = Skv;
  prm.G = Hq / Hkv;
  prm.n_qtiles = (Sq + BM - 1) / BM;
  prm.pair_heads = 1;
  prm.causal = causal ? 1 : 0;
  prm.sl2 = scale * 1.4426950408889634f;
  prm.watchdog_ns = g_watchdog_ns.load();
  const long long units = (long long)prm.n_qtiles * (Hq / 4) * B;
  if (2 * units > 0x7FFFFFFFLL) return FA_ERR_UNSUPPORTED;
  if (launch_pdl(kern, dim3((unsigned)(2 * units)), dim3(NUM_THREADS), PairLayout::REQUEST, stream, mq, mkh, mv, mo,
                 prm) != cudaSuccess) {
    (void)cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

template <int HD, bool BF16>
static int launch(const void* q, const void* k, const void* v, void* o, int hd, int B, int Hq, int Hkv, int Sq, int Skv,
                  int kv_cap, int causal, float scale, cudaStream_t stream, int dev, const Paged* pg = nullptr,
                  float* lse = nullptr) {
  if constexpr (HD == 128) {
    if (pair_applies(Hq, Hkv, pg))
      return launch_pair<BF16>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, kv_cap, causal, scale, stream, dev, lse);
  }
  // heads up to 64 wide run on the kernel with S and P in separate TMEM columns
  constexpr uint32_t REQUEST = HD == 64 ? Layout64::REQUEST : Layout<HD>::REQUEST;
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, Params);
  if constexpr (HD == 64) kern = fa_prefill64_kernel<BF16>;
  else kern = fa_prefill_kernel<HD, BF16>;
  const int slot = (HD == 128 ? 2 : 0) + (BF16 ? 1 : 0);
  if (g_attr_set[dev][slot].load() == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)REQUEST) != cudaSuccess) {
      (void)cudaGetLastError();
      return FA_ERR_SMEM;
    }
    g_attr_set[dev][slot].store(1);
  }
  EncodeTiledFn enc = encoder();
  if (!enc) return FA_ERR_LAUNCH;
  CUtensorMap mq, mk, mv, mo, mkt, mvt;
  Params prm;
  // the 128-wide kernel stores O per warp, 32 rows a box
  if (!encode_bshd(&mq, enc, q, BF16, B, Sq, Hq, hd, Sq) ||
      !encode_bshd(&mo, enc, o, BF16, B, Sq, Hq, hd, Sq, HD == 128 ? 32 : 128) ||
      !encode_kv(&mk, &mv, &mkt, &mvt, enc, k, v, BF16, B, Skv, kv_cap, Hkv, hd, pg, &prm))
    return FA_ERR_LAUNCH;
  prm.lse = lse;
  prm.o = static_cast<uint16_t*>(o);
  prm.hd = hd;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Sq = Sq;
  prm.Skv = Skv;
  prm.G = Hq / Hkv;
  prm.n_qtiles = (Sq + BM - 1) / BM;
  prm.pair_heads = (prm.G % 2 == 0) ? 1 : 0;
  prm.causal = causal ? 1 : 0;
  prm.lone_first = lone_tile_first(prm, g_dev_sms[dev].load());
  prm.sl2 = scale * 1.4426950408889634f;
  prm.watchdog_ns = g_watchdog_ns.load();
  const long long grid = grid_size(B, Hq, Hkv, Sq);
  if (launch_pdl(kern, dim3((unsigned)grid), dim3(NUM_THREADS), REQUEST, stream, mq, mk, mv, mo, mkt, mvt, prm) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

// hd = 256: one query tile per CTA (fa_prefill256_kernel).
template <bool BF16>
static int launch256(const void* q, const void* k, const void* v, void* o, int hd, int B, int Hq, int Hkv, int Sq, int Skv,
                     int kv_cap, int causal, float scale, cudaStream_t stream, int dev, float* lse = nullptr) {
  using L = Layout256;
  auto kern = fa_prefill256_kernel<BF16>;
  if (g_attr256_set[dev][BF16 ? 1 : 0].load() == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::REQUEST) != cudaSuccess) {
      (void)cudaGetLastError();
      return FA_ERR_SMEM;
    }
    g_attr256_set[dev][BF16 ? 1 : 0].store(1);
  }
  EncodeTiledFn enc = encoder();
  if (!enc) return FA_ERR_LAUNCH;
  CUtensorMap mq, mk, mv, mo;
  if (!encode_bshd(&mq, enc, q, BF16, B, Sq, Hq, hd, Sq) || !encode_bshd(&mk, enc, k, BF16, B, Skv, Hkv, hd, kv_cap) ||
      !encode_bshd(&mv, enc, v, BF16, B, Skv, Hkv, hd, kv_cap) || !encode_bshd(&mo, enc, o, BF16, B, Sq, Hq, hd, Sq))
    return FA_ERR_LAUNCH;
  Params prm;
  std::memset(&prm, 0, sizeof(prm));
  prm.o = static_cast<uint16_t*>(o);
  prm.hd = hd;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Sq = Sq;
  prm.Skv = Skv;
  prm.G = Hq / Hkv;
  prm.n_qtiles = (Sq + BM - 1) / BM;
  prm.causal = causal ? 1 : 0;
  prm.sl2 = scale * 1.4426950408889634f;
  prm.watchdog_ns = g_watchdog_ns.load();
  prm.lse = lse;
  const long long grid = (long long)prm.n_qtiles * Hq * B;
  if (grid > 0x7FFFFFFFLL) return FA_ERR_UNSUPPORTED;
  if (launch_pdl(kern, dim3((unsigned)grid), dim3(NUM_THREADS_256), L::REQUEST, stream, mq, mk, mv, mo, prm) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

// Argument checks shared by every entry point (no device call).  May replace
// k and v by q when Skv == 0 (no key is ever loaded; the maps need a base).
// The kernel a head dimension runs on: a multiple of 8 (16-byte rows for TMA)
// up to 256, on the 64, 128 or 256 kernel.  A narrower head's maps describe
// its true width, so TMA loads the missing columns of Q, K and V as zeros and
// clips them from the O store: S and P V are unchanged by the zero columns.
static int kernel_hd(int hd) {
  if (hd < 8 || hd % 8 != 0 || hd > 256) return 0;
  return hd <= 64 ? 64 : hd <= 128 ? 128 : 256;
}

static int validate(const void* q, const void*& k, const void*& v, const void* o, int B, int Hq, int Hkv, int Sq,
                    int Skv, int hd, float scale, bool* empty) {
  *empty = false;
  if (B < 0 || Sq < 0 || Skv < 0 || Hq < 1 || Hkv < 1) return FA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (kernel_hd(hd) == 0) return FA_ERR_UNSUPPORTED;
  if (B == 0 || Sq == 0) {  // nothing to compute; no pointer is read
    *empty = true;
    return FA_OK;
  }
  if (!q || !o) return FA_ERR_INVALID_ARG;
  if (Skv > 0 && (!k || !v)) return FA_ERR_INVALID_ARG;
  if (Skv == 0) k = v = q;
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
  return FA_OK;
}

static int run(bool bf16, const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int Sq,
               int Skv, int hd, int causal, float scale, void* stream) {
  bool empty = false;
  const int vs = validate(q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, scale, &empty);
  if (vs != FA_OK || empty) return vs;
  int dev = -1;
  const int ds = check_device(&dev);
  if (ds != FA_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (kernel_hd(hd) == 256)
    return bf16 ? launch256<true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev)
                : launch256<false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev);
  if (g_force_path.load() == 2) {  // the persistent kernel over whole units (testing and measurement)
    if (kernel_hd(hd) == 128)
      return bf16 ? launch_pk<128, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, nullptr, nullptr, st, dev)
                  : launch_pk<128, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, nullptr, nullptr, st, dev);
    return bf16 ? launch_pk<64, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, nullptr, nullptr, st, dev)
                : launch_pk<64, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, nullptr, nullptr, st, dev);
  }
  if (kernel_hd(hd) == 128)
    return bf16 ? launch<128, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev)
                : launch<128, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev);
  return bf16 ? launch<64, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev)
              : launch<64, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev);
}

// ------------------------------------------------------ stream-K host side

static size_t ws_bytes_for(int hd) {
  if (kernel_hd(hd) == 128) return SkLayout<128>::WS_BYTES;
  if (kernel_hd(hd) == 64) return SkLayout<64>::WS_BYTES;
  return 0;
}

// The per-CTA starting points of an even split of all (pair, KV step) steps
// over the grid.  Cached per shape: the scan over pairs runs once per shape.
struct SkSchedule {
  int key[7];
  int G;
  int su[SK_MAX_CTAS + 1];
  int sj[SK_MAX_CTAS + 1];
  // piece slots (SkParams::pf, ph) and the split pairs the merge kernel combines
  short pf[SK_MAX_CTAS];
  short ph[SK_MAX_CTAS];
  int slots;    // piece slots in use
  int n_split;  // split pairs
  int one_seg;  // every CTA runs exactly one segment
  int mu[SK_MAX_CTAS];
  short ms[SK_MAX_CTAS];
  short mn[SK_MAX_CTAS];
};

static std::mutex g_sched_mu;
static SkSchedule g_sched_cache[8];
static int g_sched_n = 0, g_sched_next = 0;

// Cost model of the schedule, in quarter KV steps: a segment (one unit, or a
// piece of one) costs its KV steps plus a fixed part for its Q load, its O
// epilogue and, for a split unit, the partial write and the merge.  Pieces
// shorter than SK_MIN_PIECE steps are not cut: the boundary moves to the
// nearer unit edge.
constexpr int SK_SEG_COST_Q = 8;  // fixed cost of a segment: two KV steps
constexpr int SK_MIN_PIECE = 2;

// Pieces of one pair per CTA (as many pairs as CTAs or fewer): pair u is cut
// into k_u pieces of near-equal length, the next CTA always going to the pair
// whose pieces are longest, and no piece is shorter than SK_MIN_PIECE steps.
// Every CTA then runs a single segment.
static int pieces_schedule(const std::vector<int>& n, int gmax, SkSchedule* sc) {
  const int nu = static_cast<int>(n.size());
  std::vector<int> k(static_cast<size_t>(nu), 1);
  for (int left = gmax - nu; left > 0; --left) {
    int best = -1;
    long long best_len = -1;
    for (int u = 0; u < nu; ++u) {
      if (n[u] / (k[u] + 1) < SK_MIN_PIECE) continue;
      const long long len = (n[u] + k[u] - 1) / k[u];
      if (len > best_len) {
        best_len = len;
        best = u;
      }
    }
    if (best < 0) break;
    ++k[best];
  }
  int G = 0;
  for (int u = 0; u < nu; ++u)
    for (int i = 0; i < k[u]; ++i) {
      sc->su[G] = u;
      sc->sj[G] = static_cast<int>(static_cast<long long>(n[u]) * i / k[u]);
      ++G;
    }
  return G;
}

static void make_schedule(const Params& prm, int sms, SkSchedule* sc) {
  const long long nu = unit_count_of(prm);
  std::vector<int> n(static_cast<size_t>(nu));
  long long T = 0;  // total cost, quarter steps
  for (long long u = 0; u < nu; ++u) {
    n[u] = unit_geo(prm, static_cast<int>(u)).n;
    T += 4LL * n[u] + SK_SEG_COST_Q;
  }
  const int gmax = std::max(1, std::min(sms, SK_MAX_CTAS));
  const int want = static_cast<int>(std::max<long long>(1, std::min<long long>(gmax, nu * 64)));
  int G = 1;
  sc->su[0] = 0;
  sc->sj[0] = 0;
  sc->one_seg = nu <= gmax ? 1 : 0;
  if (sc->one_seg) G = pieces_schedule(n, gmax, sc);
  // otherwise CTA c starts at cost T c / want, rounded to a (unit, step)
  // boundary; boundaries strictly increase, so no CTA's range is empty
  long long acc = 0;  // cost of units [0, u)
  int u = 0;
  for (int c = 1; !sc->one_seg && c < want; ++c) {
    const long long target = T * c / want;
    while (u < nu && acc + 4LL * n[u] + SK_SEG_COST_Q <= target) acc += 4LL * n[u++] + SK_SEG_COST_Q;
    if (u >= nu) break;
    const long long j = (target - acc - SK_SEG_COST_Q) / 4;  // KV steps into unit u (may be negative)
    int bu = u, bj;
    if (j < SK_MIN_PIECE) {
      bj = 0;
    } else if (n[u] - j < SK_MIN_PIECE) {
      bu = u + 1;
      bj = 0;
    } else {
      bj = static_cast<int>(j);
    }
    if (bu >= nu) break;
    if (bu > sc->su[G - 1] || (bu == sc->su[G - 1] && bj > sc->sj[G - 1])) {
      sc->su[G] = bu;
      sc->sj[G] = bj;
      ++G;
    }
  }
  sc->G = G;
  sc->su[G] = static_cast<int>(nu);
  sc->sj[G] = 0;
  // Piece slots, in CTA order: a CTA that starts inside a pair continues the
  // pair opened last (its first segment gets the next slot); a CTA whose range
  // ends inside a pair it entered at KV tile 0 opens that pair (its last
  // segment gets the next slot).  So every split pair's pieces hold
  // consecutive slots in KV order, the piece with KV tile 0 first.
  int slot = 0, ns = 0;
  for (int c = 0; c < G; ++c) {
    sc->pf[c] = sc->ph[c] = -1;
    if (sc->sj[c] > 0 && ns > 0 && sc->mu[ns - 1] == sc->su[c]) {
      sc->pf[c] = static_cast<short>(slot++);
      ++sc->mn[ns - 1];
    }
    const bool ends_inside = sc->sj[c + 1] > 0;
    const bool single_tail = sc->su[c + 1] == sc->su[c] && sc->sj[c] > 0;  // one segment, not at tile 0
    if (ends_inside && !single_tail) {
      sc->ph[c] = static_cast<short>(slot++);
      sc->mu[ns] = sc->su[c + 1];
      sc->ms[ns] = sc->ph[c];
      sc->mn[ns] = 1;
      ++ns;
    }
  }
  sc->slots = slot;
  sc->n_split = ns;
}

static void get_schedule(const Params& prm, int sms, SkSchedule* out) {
  const int key[7] = {prm.B, prm.Hq, prm.Hkv, prm.Sq, prm.Skv, prm.causal, sms};
  std::lock_guard<std::mutex> lk(g_sched_mu);
  for (int i = 0; i < g_sched_n; ++i)
    if (std::memcmp(g_sched_cache[i].key, key, sizeof(key)) == 0) {
      *out = g_sched_cache[i];
      return;
    }
  SkSchedule& sc = g_sched_cache[g_sched_next];
  std::memcpy(sc.key, key, sizeof(key));
  make_schedule(prm, sms, &sc);
  *out = sc;
  g_sched_next = (g_sched_next + 1) % 8;
  if (g_sched_n < 8) ++g_sched_n;
}

// The split pairs' merge, after the stream-K kernel on the same stream
// (programmatic dependent launch: it waits for every piece).
template <int HD, bool BF16>
static int launch_merge(const SkSchedule& sc, const Params& prm, const float4* ws_o, const float* ws_ml,
                        cudaStream_t stream) {
  if (sc.n_split == 0) return FA_OK;
  MergeParams mp;
  std::memset(&mp, 0, sizeof(mp));
  mp.p = prm;
  mp.ws_o = ws_o;
  mp.ws_ml = ws_ml;
  mp.n_split = sc.n_split;
  std::memcpy(mp.mu, sc.mu, sizeof(int) * sc.n_split);
  std::memcpy(mp.ms, sc.ms, sizeof(short) * sc.n_split);
  std::memcpy(mp.mn, sc.mn, sizeof(short) * sc.n_split);
  const unsigned grid = static_cast<unsigned>(sc.n_split) * 2u * (BM / 32) * (HD / 64);
  if (launch_pdl(fa_sk_merge_kernel<HD, BF16>, dim3(grid), dim3(MERGE_THREADS), 0, stream, mp) != cudaSuccess) {
    (void)cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

// Opt one stream-K instantiation in to its shared memory, once per device.
template <typename K>
static bool sk_attr(K kern, int dev, int slot, uint32_t bytes) {
  if (g_sk_attr_set[dev][slot].load() != 0) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  g_sk_attr_set[dev][slot].store(1);
  return true;
}

template <int HD, bool BF16>
static int launch_sk(const void* q, const void* k, const void* v, void* o, int hd, int B, int Hq, int Hkv, int Sq, int Skv,
                     int kv_cap, int causal, float scale, void* ws, cudaStream_t stream, int dev,
                     const Paged* pg = nullptr, float* lse = nullptr) {
  using SL = SkLayout<HD>;
  EncodeTiledFn enc = encoder();
  if (!enc) return FA_ERR_LAUNCH;
  CUtensorMap mq, mk, mv, mo, mkt, mvt;
  Params pkv;
  if (!encode_bshd(&mq, enc, q, BF16, B, Sq, Hq, hd, Sq) || !encode_bshd(&mo, enc, o, BF16, B, Sq, Hq, hd, Sq) ||
      !encode_kv(&mk, &mv, &mkt, &mvt, enc, k, v, BF16, B, Skv, kv_cap, Hkv, hd, pg, &pkv))
    return FA_ERR_LAUNCH;
  SkParams sp;
  std::memset(&sp, 0, sizeof(sp));
  Params& prm = sp.p;
  prm.o = static_cast<uint16_t*>(o);
  prm.hd = hd;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Sq = Sq;
  prm.Skv = Skv;
  prm.G = Hq / Hkv;
  prm.n_qtiles = (Sq + BM - 1) / BM;
  prm.pair_heads = (prm.G % 2 == 0) ? 1 : 0;
  prm.causal = causal ? 1 : 0;
  prm.lone_first = 1;  // split-KV: fewer steps in total
  prm.sl2 = scale * 1.4426950408889634f;
  prm.block_table = pkv.block_table;
  prm.page_size = pkv.page_size;
  prm.max_pages = pkv.max_pages;
  prm.num_blocks = pkv.num_blocks;
  prm.last_page = pkv.last_page;
  prm.lse = lse;
  prm.watchdog_ns = g_watchdog_ns.load();
  SkSchedule sc;
  get_schedule(prm, g_dev_sms[dev].load(), &sc);
  uint8_t* base = static_cast<uint8_t*>(ws);
  sp.ws_o = reinterpret_cast<float4*>(base);
  sp.ws_ml = reinterpret_cast<float*>(base + SL::WS_O_BYTES);
  // CTAs that run several segments: the persistent kernel (its epilogue
  // warpgroup overlaps each segment's output with the next segment's steps)
  if (!sc.one_seg || g_force_path.load() == 2)
    return launch_pk<HD, BF16>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, kv_cap, causal, scale, sp.ws_o, sp.ws_ml, stream, dev,
                               pg, lse);
  auto kern = fa_prefill_sk_kernel<HD, BF16>;
  if (!sk_attr(kern, dev, (HD == 128 ? 2 : 0) + (BF16 ? 1 : 0), SL::REQUEST)) return FA_ERR_SMEM;
  std::memcpy(sp.su, sc.su, sizeof(int) * (sc.G + 1));
  std::memcpy(sp.sj, sc.sj, sizeof(int) * (sc.G + 1));
  std::memcpy(sp.pf, sc.pf, sizeof(short) * sc.G);
  std::memcpy(sp.ph, sc.ph, sizeof(short) * sc.G);
  if (launch_pdl(kern, dim3(static_cast<unsigned>(sc.G)), dim3(NUM_THREADS), SL::REQUEST, stream, mq, mk, mv, mo, mkt,
                 mvt, sp) != cudaSuccess) {
    (void)cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return launch_merge<HD, BF16>(sc, prm, sp.ws_o, sp.ws_ml, stream);
}

// The persistent kernel.  Without a workspace (ws_o == nullptr) every CTA
// takes whole units in snake order (grid = min(SMs, units)); with one, the
// stream-K ranges of the split-KV schedule, then the merge of the split units.
template <int HD, bool BF16>
static int launch_pk(const void* q, const void* k, const void* v, void* o, int hd, int B, int Hq, int Hkv, int Sq, int Skv,
                     int kv_cap, int causal, float scale, float4* ws_o, float* ws_ml, cudaStream_t stream, int dev,
                     const Paged* pg, float* lse) {
  using PL = PkLayout<HD>;
  EncodeTiledFn enc = encoder();
  if (!enc) return FA_ERR_LAUNCH;
  CUtensorMap mq, mk, mv, mkt, mvt;
  Params pkv;
  if (!encode_bshd(&mq, enc, q, BF16, B, Sq, Hq, hd, Sq) ||
      !encode_kv(&mk, &mv, &mkt, &mvt, enc, k, v, BF16, B, Skv, kv_cap, Hkv, hd, pg, &pkv))
    return FA_ERR_LAUNCH;
  PkParams sp;
  std::memset(&sp, 0, sizeof(sp));
  Params& prm = sp.p;
  prm.o = static_cast<uint16_t*>(o);
  prm.hd = hd;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Sq = Sq;
  prm.Skv = Skv;
  prm.G = Hq / Hkv;
  prm.n_qtiles = (Sq + BM - 1) / BM;
  prm.pair_heads = (prm.G % 2 == 0) ? 1 : 0;
  prm.causal = causal ? 1 : 0;
  prm.lone_first = ws_o ? 1 : lone_tile_first(prm, g_dev_sms[dev].load());  // split-KV: fewer steps in total
  prm.sl2 = scale * 1.4426950408889634f;
  prm.block_table = pkv.block_table;
  prm.page_size = pkv.page_size;
  prm.max_pages = pkv.max_pages;
  prm.num_blocks = pkv.num_blocks;
  prm.last_page = pkv.last_page;
  prm.lse = lse;
  prm.watchdog_ns = g_watchdog_ns.load();
  const long long nu = unit_count_of(prm);
  if (nu > 0x7FFFFFFFLL) return FA_ERR_UNSUPPORTED;
  sp.n_units = static_cast<int>(nu);
  const int sms = g_dev_sms[dev].load();
  auto kern = fa_prefill_pk_kernel<HD, BF16>;
  const int aslot = (HD == 128 ? 2 : 0) + (BF16 ? 1 : 0);
  if (g_pk_attr_set[dev][aslot].load() == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PL::REQUEST) != cudaSuccess) {
      (void)cudaGetLastError();
      return FA_ERR_SMEM;
    }
    g_pk_attr_set[dev][aslot].store(1);
  }
  SkSchedule sc;
  int grid;
  if (ws_o) {
    get_schedule(prm, sms, &sc);
    sp.ranges = 1;
    grid = sc.G;
    std::memcpy(sp.su, sc.su, sizeof(int) * (sc.G + 1));
    std::memcpy(sp.sj, sc.sj, sizeof(int) * (sc.G + 1));
    std::memcpy(sp.pf, sc.pf, sizeof(short) * sc.G);
    std::memcpy(sp.ph, sc.ph, sizeof(short) * sc.G);
    sp.ws_o = ws_o;
    sp.ws_ml = ws_ml;
  } else {
    sp.ranges = 0;
    grid = static_cast<int>(std::min<long long>(nu, std::max(1, sms)));
  }
  if (launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(PK_THREADS), PL::REQUEST, stream, mq, mk, mv, mkt, mvt,
                 sp) != cudaSuccess) {
    (void)cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return ws_o ? launch_merge<HD, BF16>(sc, prm, sp.ws_o, sp.ws_ml, stream) : FA_OK;
}

// Attention over a K/V cache of kv_cap rows per sequence of which the first
// kv_len are valid: the maps describe kv_len rows with a batch stride of
// kv_cap, so rows past kv_len (stale or unwritten cache) load as zeros.
static int run_kvcache(bool bf16, const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
                       int Sq, int kv_len, int kv_cap, int hd, int causal, float scale, void* ws, size_t ws_bytes,
                       void* stream) {
  if (kv_len < 0 || kv_cap < 0 || kv_len > kv_cap) return FA_ERR_INVALID_ARG;
  bool empty = false;
  const int vs = validate(q, k, v, o, B, Hq, Hkv, Sq, kv_len, hd, scale, &empty);
  if (vs != FA_OK || empty) return vs;
  if ((long long)kv_cap > 0x7FFFFFFFLL - 256 || (unsigned long long)kv_cap * Hkv * hd * 2 >= (1ull << 40))
    return FA_ERR_UNSUPPORTED;
  const unsigned long long qn = (unsigned long long)B * Sq * Hq * hd;
  const unsigned long long cn = (unsigned long long)B * kv_cap * Hkv * hd;
  if (kv_len > 0 && (overlaps(o, qn * 2, k, cn * 2) || overlaps(o, qn * 2, v, cn * 2))) return FA_ERR_INVALID_ARG;
  if (ws) {
    if (kernel_hd(hd) == 256) return FA_ERR_UNSUPPORTED;  // split-KV: heads up to 128 wide
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return FA_ERR_ALIGNMENT;
    if (ws_bytes < ws_bytes_for(hd)) return FA_ERR_INVALID_ARG;
  }
  int dev = -1;
  const int ds = check_device(&dev);
  if (ds != FA_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int stride = kv_len > 0 ? kv_cap : 0;  // kv_len == 0: the maps point at q (no key is loaded)
  if (kernel_hd(hd) == 256)
    return bf16 ? launch256<true>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, stride, causal, scale, st, dev)
                : launch256<false>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, stride, causal, scale, st, dev);
  if (ws) {
    if (kernel_hd(hd) == 128)
      return bf16 ? launch_sk<128, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, stride, causal, scale, ws, st, dev)
                  : launch_sk<128, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, stride, causal, scale, ws, st, dev);
    return bf16 ? launch_sk<64, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, stride, causal, scale, ws, st, dev)
                : launch_sk<64, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, stride, causal, scale, ws, st, dev);
  }
  if (kernel_hd(hd) == 128)
    return bf16 ? launch<128, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, stride, causal, scale, st, dev)
                : launch<128, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, stride, causal, scale, st, dev);
  return bf16 ? launch<64, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, stride, causal, scale, st, dev)
              : launch<64, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, stride, causal, scale, st, dev);
}

// Attention over a paged K/V pool (one-shot kernel).
static int run_paged(bool bf16, const void* q, const void* k_pool, const void* v_pool, const void* block_table,
                     void* o, int B, int Hq, int Hkv, int Sq, int kv_len, int hd, int page_size, int max_pages,
                     int num_blocks, int causal, float scale, void* ws, size_t ws_bytes, void* stream) {
  if (kv_len < 0 || page_size < BN || page_size % BN != 0 || max_pages < 0 || num_blocks < 1)
    return FA_ERR_INVALID_ARG;
  if ((long long)max_pages * page_size < kv_len) return FA_ERR_INVALID_ARG;
  bool empty = false;
  const void* k = k_pool;
  const void* v = v_pool;
  const int vs = validate(q, k, v, o, B, Hq, Hkv, Sq, kv_len, hd, scale, &empty);
  if (vs != FA_OK || empty) return vs;
  if (kernel_hd(hd) == 256) return FA_ERR_UNSUPPORTED;  // heads over 128 wide: the one-shot kernel only
  if (kv_len > 0) {
    if (!block_table) return FA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(block_table) & 3u) return FA_ERR_ALIGNMENT;
    if ((unsigned long long)page_size * Hkv * hd * 2 >= (1ull << 40)) return FA_ERR_UNSUPPORTED;
    const unsigned long long qn = (unsigned long long)B * Sq * Hq * hd;
    const unsigned long long pn = (unsigned long long)num_blocks * page_size * Hkv * hd;
    if (overlaps(o, qn * 2, k, pn * 2) || overlaps(o, qn * 2, v, pn * 2) ||
        overlaps(o, qn * 2, block_table, (size_t)B * max_pages * 4))
      return FA_ERR_INVALID_ARG;
  }
  int dev = -1;
  const int ds = check_device(&dev);
  if (ds != FA_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Paged pg{static_cast<const int*>(block_table), page_size, max_pages, num_blocks};
  if (ws) {  // split-KV over the pool
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return FA_ERR_ALIGNMENT;
    if (ws_bytes < ws_bytes_for(hd)) return FA_ERR_INVALID_ARG;
    if (kernel_hd(hd) == 128)
      return bf16 ? launch_sk<128, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, kv_len, causal, scale, ws, st, dev, &pg)
                  : launch_sk<128, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, kv_len, causal, scale, ws, st, dev, &pg);
    return bf16 ? launch_sk<64, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, kv_len, causal, scale, ws, st, dev, &pg)
                : launch_sk<64, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, kv_len, causal, scale, ws, st, dev, &pg);
  }
  if (kernel_hd(hd) == 128)
    return bf16 ? launch<128, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, kv_len, causal, scale, st, dev, &pg)
                : launch<128, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, kv_len, causal, scale, st, dev, &pg);
  return bf16 ? launch<64, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, kv_len, causal, scale, st, dev, &pg)
              : launch<64, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, kv_len, kv_len, causal, scale, st, dev, &pg);
}

// Any supported hd, either kernel (a workspace selects split-KV), and an
// optional per-row log-sum-exp output.
static int run_ex(bool bf16, const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                  int Hkv, int Sq, int Skv, int hd, int causal, float scale, void* ws, size_t ws_bytes, void* stream) {
  bool empty = false;
  const int vs = validate(q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, scale, &empty);
  if (vs != FA_OK || empty) return vs;
  if (lse) {
    if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_ALIGNMENT;
    const size_t ln = (size_t)B * Hq * Sq * 4, qn = (size_t)B * Sq * Hq * hd * 2, kn = (size_t)B * Skv * Hkv * hd * 2;
    if (overlaps(lse, ln, q, qn) || overlaps(lse, ln, o, qn) || (Skv > 0 && (overlaps(lse, ln, k, kn) || overlaps(lse, ln, v, kn))))
      return FA_ERR_INVALID_ARG;
  }
  if (ws) {
    if (kernel_hd(hd) == 256) return FA_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return FA_ERR_ALIGNMENT;
    if (ws_bytes < ws_bytes_for(hd)) return FA_ERR_INVALID_ARG;
    if (lse && overlaps(lse, (size_t)B * Hq * Sq * 4, ws, ws_bytes)) return FA_ERR_INVALID_ARG;
  }
  int dev = -1;
  const int ds = check_device(&dev);
  if (ds != FA_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (kernel_hd(hd) == 256)
    return bf16 ? launch256<true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev, lse)
                : launch256<false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev, lse);
  if (ws) {
    if (kernel_hd(hd) == 128)
      return bf16 ? launch_sk<128, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, ws, st, dev, nullptr, lse)
                  : launch_sk<128, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, ws, st, dev, nullptr, lse);
    return bf16 ? launch_sk<64, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, ws, st, dev, nullptr, lse)
                : launch_sk<64, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, ws, st, dev, nullptr, lse);
  }
  if (kernel_hd(hd) == 128)
    return bf16 ? launch<128, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev, nullptr, lse)
                : launch<128, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev, nullptr, lse);
  return bf16 ? launch<64, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev, nullptr, lse)
              : launch<64, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev, nullptr, lse);
}

static int run_ws(bool bf16, const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int Sq,
                  int Skv, int hd, int causal, float scale, void* ws, size_t ws_bytes, void* stream) {
  bool empty = false;
  const int vs = validate(q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, scale, &empty);
  if (vs != FA_OK || empty) return vs;
  if (kernel_hd(hd) == 256) return FA_ERR_UNSUPPORTED;  // heads over 128 wide: the one-shot kernel only
  if (!ws) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return FA_ERR_ALIGNMENT;
  if (ws_bytes < ws_bytes_for(hd)) return FA_ERR_INVALID_ARG;
  int dev = -1;
  const int ds = check_device(&dev);
  if (ds != FA_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (g_force_path.load() == 1) {
    if (kernel_hd(hd) == 128)
      return bf16 ? launch<128, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev)
                  : launch<128, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev);
    return bf16 ? launch<64, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev)
                : launch<64, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, st, dev);
  }
  if (kernel_hd(hd) == 128)
    return bf16 ? launch_sk<128, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, ws, st, dev)
                : launch_sk<128, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, ws, st, dev);
  return bf16 ? launch_sk<64, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, ws, st, dev)
              : launch_sk<64, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, Skv, causal, scale, ws, st, dev);
}

}  // namespace fa

#include "kv_append.cuh"

namespace fa {

// ==================================== split-KV with library-owned scratch
//
// fa_prefill_ws_static: the split-KV kernel and schedule above, unchanged,
// with its scratch in a file-scope device array instead of a caller
// workspace.  It serves callers that cannot allocate device memory when they
// call: an engine whose device memory is laid out once at start-up and may
// not grow per request (an allocation at peak load can fail, or stall on the
// allocator), and a C host with no device allocator of its own that holds
// only the tensors it is given.  Nothing here allocates or frees device
// memory.  Layout of the array (the kernel indexes every region by CTA slot):
//   [0, 1 MB)         m and l: 512 piece slots x 2 tiles x 2 x 128 f32
//   [1 MB, ...)       partial O: (the call's piece slots) x 2 x 128 x hd f32
static __device__ __align__(256) unsigned char g_static_scratch[FA_STATIC_SCRATCH_BYTES];

constexpr size_t STATIC_ML_BYTES = (size_t)SK_SLOTS * 2 * 2 * BM * 4;
constexpr size_t STATIC_O_OFF = STATIC_ML_BYTES;
static_assert(STATIC_O_OFF % 256 == 0, "region alignment");
static_assert(STATIC_O_OFF + (size_t)2 * SK_MAX_CTAS * 2 * BM * 64 * 4 <= FA_STATIC_SCRATCH_BYTES,
              "two pieces per CTA of a full grid must fit at hd 64");

static size_t static_bytes_needed(int hd, int slots) { return STATIC_O_OFF + (size_t)slots * 2 * BM * hd * 4; }

static std::mutex g_static_mu;
static uint8_t* g_static_base[MAX_DEVICES];

// The array's device address, looked up once per device (the first call);
// no part of it needs initialising (every slot a call reads, that call's
// stream-K kernel has written).
static int static_scratch(int dev, cudaStream_t stream, uint8_t** base) {
  (void)stream;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (g_static_base[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return FA_ERR_DEVICE;
    }
    g_static_base[dev] = static_cast<uint8_t*>(p);
  }
  *base = g_static_base[dev];
  return FA_OK;
}

template <int HD, bool BF16>
static int launch_sk_static(const void* q, const void* k, const void* v, void* o, int hd, int B, int Hq, int Hkv, int Sq,
                            int Skv, int causal, float scale, uint8_t* base, cudaStream_t stream, int dev) {
  const int kv_cap = Skv;
  using SL = SkLayout<HD>;
  SkParams sp;
  std::memset(&sp, 0, sizeof(sp));
  Params& prm = sp.p;
  prm.o = static_cast<uint16_t*>(o);
  prm.hd = hd;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Sq = Sq;
  prm.Skv = Skv;
  prm.G = Hq / Hkv;
  prm.n_qtiles = (Sq + BM - 1) / BM;
  prm.pair_heads = (prm.G % 2 == 0) ? 1 : 0;
  prm.causal = causal ? 1 : 0;
  prm.lone_first = 1;  // split-KV: fewer steps in total
  prm.sl2 = scale * 1.4426950408889634f;
  prm.watchdog_ns = g_watchdog_ns.load();
  SkSchedule sc;
  get_schedule(prm, g_dev_sms[dev].load(), &sc);
  if (static_bytes_needed(HD, sc.slots) > FA_STATIC_SCRATCH_BYTES) return FA_ERR_SCRATCH;
  std::memcpy(sp.su, sc.su, sizeof(int) * (sc.G + 1));
  std::memcpy(sp.sj, sc.sj, sizeof(int) * (sc.G + 1));
  std::memcpy(sp.pf, sc.pf, sizeof(short) * sc.G);
  std::memcpy(sp.ph, sc.ph, sizeof(short) * sc.G);
  sp.ws_ml = reinterpret_cast<float*>(base);
  sp.ws_o = reinterpret_cast<float4*>(base + STATIC_O_OFF);
  if (!sc.one_seg)  // as the workspace path: multi-segment CTAs on the persistent kernel
    return launch_pk<HD, BF16>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, kv_cap, causal, scale, sp.ws_o, sp.ws_ml, stream, dev);
  auto kern = fa_prefill_sk_kernel<HD, BF16>;
  if (!sk_attr(kern, dev, (HD == 128 ? 2 : 0) + (BF16 ? 1 : 0), SL::REQUEST)) return FA_ERR_SMEM;
  EncodeTiledFn enc = encoder();
  if (!enc) return FA_ERR_LAUNCH;
  // the maps describe the caller's head width hd (<= HD): TMA zero-fills the
  // missing columns and never reads past the tensors
  CUtensorMap mq, mk, mv, mo, mkt, mvt;
  Params pkv;
  if (!encode_bshd(&mq, enc, q, BF16, B, Sq, Hq, hd, Sq) || !encode_bshd(&mo, enc, o, BF16, B, Sq, Hq, hd, Sq) ||
      !encode_kv(&mk, &mv, &mkt, &mvt, enc, k, v, BF16, B, Skv, kv_cap, Hkv, hd, nullptr, &pkv))
    return FA_ERR_LAUNCH;
  if (launch_pdl(kern, dim3(static_cast<unsigned>(sc.G)), dim3(NUM_THREADS), SL::REQUEST, stream, mq, mk, mv, mo, mkt,
                 mvt, sp) != cudaSuccess) {
    (void)cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return launch_merge<HD, BF16>(sc, prm, sp.ws_o, sp.ws_ml, stream);
}

static int run_static(bool bf16, const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
                      int Sq, int Skv, int hd, int causal, float scale, void* stream) {
  bool empty = false;
  const int vs = validate(q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, scale, &empty);
  if (vs != FA_OK || empty) return vs;
  if (kernel_hd(hd) == 256) return FA_ERR_UNSUPPORTED;  // heads over 128 wide: the one-shot kernel only
  int dev = -1;
  const int ds = check_device(&dev);
  if (ds != FA_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* base = nullptr;
  const int ss = static_scratch(dev, st, &base);
  if (ss != FA_OK) return ss;
  if (kernel_hd(hd) == 128)
    return bf16 ? launch_sk_static<128, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, causal, scale, base, st, dev)
                : launch_sk_static<128, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, causal, scale, base, st, dev);
  return bf16 ? launch_sk_static<64, true>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, causal, scale, base, st, dev)
              : launch_sk_static<64, false>(q, k, v, o, hd, B, Hq, Hkv, Sq, Skv, causal, scale, base, st, dev);
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

extern "C" int fa_prefill_ws(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int Sq,
                             int Skv, int hd, int causal, float scale, void* workspace, size_t workspace_bytes,
                             void* stream) {
  return fa::run_ws(false, q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, causal, scale, workspace, workspace_bytes, stream);
}

extern "C" int fa_prefill_ws_bf16(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
                                  int Sq, int Skv, int hd, int causal, float scale, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return fa::run_ws(true, q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, causal, scale, workspace, workspace_bytes, stream);
}

extern "C" size_t fa_workspace_bytes(int hd) { return fa::ws_bytes_for(hd); }

extern "C" int fa_prefill_kvcache(const void* q, const void* k_cache, const void* v_cache, void* o, int B, int Hq,
                                  int Hkv, int Sq, int kv_len, int kv_cap, int hd, int causal, float scale, int bf16,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  return fa::run_kvcache(bf16 != 0, q, k_cache, v_cache, o, B, Hq, Hkv, Sq, kv_len, kv_cap, hd, causal, scale,
                         workspace, workspace_bytes, stream);
}

extern "C" int fa_prefill_paged(const void* q, const void* k_pool, const void* v_pool, const void* block_table,
                                void* o, int B, int Hq, int Hkv, int Sq, int kv_len, int hd, int page_size,
                                int max_pages, int num_blocks, int causal, float scale, int bf16, void* stream) {
  return fa::run_paged(bf16 != 0, q, k_pool, v_pool, block_table, o, B, Hq, Hkv, Sq, kv_len, hd, page_size,
                       max_pages, num_blocks, causal, scale, nullptr, 0, stream);
}

extern "C" int fa_prefill_paged_ws(const void* q, const void* k_pool, const void* v_pool, const void* block_table,
                                   void* o, int B, int Hq, int Hkv, int Sq, int kv_len, int hd, int page_size,
                                   int max_pages, int num_blocks, int causal, float scale, int bf16, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  if (!workspace) return FA_ERR_INVALID_ARG;
  return fa::run_paged(bf16 != 0, q, k_pool, v_pool, block_table, o, B, Hq, Hkv, Sq, kv_len, hd, page_size,
                       max_pages, num_blocks, causal, scale, workspace, workspace_bytes, stream);
}

extern "C" int fa_kv_append(const void* k_new, const void* v_new, const void* positions, void* k_cache, void* v_cache,
                            int B, int T, int Hkv, int hd, int kv_cap, int bf16, void* stream) {
  return fa::run_kv_append(k_new, v_new, positions, k_cache, v_cache, B, T, Hkv, hd, kv_cap, bf16 != 0, stream);
}

extern "C" int fa_prefill_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                             int Hkv, int Sq, int Skv, int hd, int causal, float scale, int bf16, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return fa::run_ex(bf16 != 0, q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, hd, causal, scale, workspace, workspace_bytes,
                    stream);
}

namespace fa {

// The one-shot grid's wave efficiency: its pairs run longest first in waves
// of `sms`, so each wave lasts as long as its first (longest) pair; the
// efficiency is the pairs' KV steps over sms x that sum.  Host-only.
static double oneshot_wave_efficiency(int B, int Hq, int Hkv, int Sq, int Skv, int causal, int sms) {
  Params prm;
  std::memset(&prm, 0, sizeof(prm));
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Sq = Sq;
  prm.Skv = Skv;
  prm.G = Hq / Hkv;
  prm.n_qtiles = (Sq + BM - 1) / BM;
  prm.pair_heads = (prm.G % 2 == 0) ? 1 : 0;
  prm.causal = causal ? 1 : 0;
  prm.lone_first = lone_tile_first(prm, sms);  // the one-shot grid's pairing
  const long long nu = unit_count_of(prm);
  long long total = 0, makespan = 0;
  for (long long u = 0; u < nu; ++u) {
    const int n = unit_geo(prm, static_cast<int>(u)).n;
    total += n;
    if (u % sms == 0) makespan += n;
  }
  return makespan > 0 ? static_cast<double>(total) / (static_cast<double>(sms) * makespan) : 1.0;
}

static int split_advice(int B, int Hq, int Hkv, int Sq, int Skv, int hd, int causal) {
  if (B < 0 || Sq < 0 || Skv < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return -FA_ERR_INVALID_ARG;
  if (hd != 0 && kernel_hd(hd) == 0) return -FA_ERR_UNSUPPORTED;
  if (B == 0 || Sq == 0 || Skv == 0) return 0;
  if (hd > 128) return 0;  // split-KV takes heads up to 128 wide
  int dev = -1;
  const int ds = check_device(&dev);
  if (ds != FA_OK) return -ds;
  const long long units = grid_size(B, Hq, Hkv, Sq);
  const long long longest = (Skv + BN - 1) / BN;
  const long long sms = g_dev_sms[dev].load();
  // an underfilled one-shot grid with long rows (causal or not, the longest
  // query tile walks all Skv keys under the bottom-right alignment)
  if (2 * units <= sms && longest >= 8) return 1;
  // hd 64: more pairs than SMs, but whole waves of them leave SMs idle --
  // the persistent kernel's stream-K ranges even the load out.  At hd 64 its
  // whole call (step rate, splits, merge) costs ~1.18x the work of the
  // one-shot kernel's busy time (chunked prefill: 133.1 us against 135.3 us at
  // a wave efficiency of 0.835), so it pays below ~0.85; at hd 128 its step is
  // 10-15 % slower, more than the quantization it removes
  if (hd != 0 && kernel_hd(hd) == 64 && units > sms && units <= (1 << 20) &&
      oneshot_wave_efficiency(B, Hq, Hkv, Sq, Skv, causal, static_cast<int>(sms)) < 0.85)
    return 1;
  return 0;
}

}  // namespace fa

extern "C" int fa_split_kv_advised(int B, int Hq, int Hkv, int Sq, int Skv, int causal) {
  return fa::split_advice(B, Hq, Hkv, Sq, Skv, 0, causal);
}

extern "C" int fa_split_kv_advised_hd(int B, int Hq, int Hkv, int Sq, int Skv, int hd, int causal) {
  return fa::split_advice(B, Hq, Hkv, Sq, Skv, hd, causal);
}

extern "C" int fa_prefill_ws_static(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
                                    int Sq, int Skv, int hd, int causal, float scale, int bf16, void* stream) {
  return fa::run_static(bf16 != 0, q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, causal, scale, stream);
}

extern "C" const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null pointer, bad size, Hq % Hkv != 0, bad scale or aliasing";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: hd must be a multiple of 8 up to 256 (split-KV and paged: up to 128) and tensors must fit TMA coordinates";
    case FA_ERR_ALIGNMENT: return "FA_ERR_ALIGNMENT: q, k, v and o must be 16-byte aligned";
    case FA_ERR_SMEM: return "FA_ERR_SMEM: shared-memory request does not fit the device";
    case FA_ERR_LAUNCH: return "FA_ERR_LAUNCH: TMA descriptor encode or kernel launch failed";
    case FA_ERR_DEVICE: return "FA_ERR_DEVICE: no current device or not an sm_103 GPU";
    case FA_ERR_SCRATCH: return "FA_ERR_SCRATCH: the call needs more than the static scratch maximum (FA_STATIC_SCRATCH_BYTES)";
    default: return "unknown fa_status_t";
  }
}

extern "C" int fa_debug_schedule(int B, int Hq, int Hkv, int Sq, int Skv, int causal, int sms, int* cta_pair,
                                 int* cta_step, int* pair_steps, int max_pairs, int* out) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Sq < 1 || Skv < 1 || sms < 1 || !cta_pair || !cta_step || !out)
    return -FA_ERR_INVALID_ARG;
  fa::Params prm;
  std::memset(&prm, 0, sizeof(prm));
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Sq = Sq;
  prm.Skv = Skv;
  prm.G = Hq / Hkv;
  prm.n_qtiles = (Sq + fa::BM - 1) / fa::BM;
  prm.pair_heads = (prm.G % 2 == 0) ? 1 : 0;
  prm.causal = causal ? 1 : 0;
  prm.lone_first = 1;  // as the split-KV path
  const long long nu = fa::unit_count_of(prm);
  if (nu > 0x7FFFFFFF) return -FA_ERR_UNSUPPORTED;
  if (pair_steps && nu > max_pairs) return -FA_ERR_UNSUPPORTED;
  fa::SkSchedule sc;
  fa::make_schedule(prm, sms, &sc);
  for (int c = 0; c <= sc.G; ++c) {
    cta_pair[c] = sc.su[c];
    cta_step[c] = sc.sj[c];
  }
  if (pair_steps)
    for (long long u = 0; u < nu; ++u) pair_steps[u] = fa::unit_geo(prm, static_cast<int>(u)).n;
  out[0] = sc.G;
  out[1] = sc.one_seg;
  out[2] = sc.n_split;
  out[3] = sc.slots;
  return static_cast<int>(nu);
}

extern "C" int fa_debug_row_pairing(int B, int Hq, int Hkv, int Sq, int Skv, int causal, int sms) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Sq < 1 || Skv < 1 || sms < 1) return -FA_ERR_INVALID_ARG;
  fa::Params prm;
  std::memset(&prm, 0, sizeof(prm));
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Sq = Sq;
  prm.Skv = Skv;
  prm.G = Hq / Hkv;
  prm.n_qtiles = (Sq + fa::BM - 1) / fa::BM;
  prm.pair_heads = (prm.G % 2 == 0) ? 1 : 0;
  prm.causal = causal ? 1 : 0;
  return fa::lone_tile_first(prm, sms);
}

extern "C" unsigned int fa_smem_bytes(int hd) {
  if (fa::kernel_hd(hd) == 256) return fa::Layout256::REQUEST;
  if (fa::kernel_hd(hd) == 128) return fa::Layout<128>::REQUEST;
  if (fa::kernel_hd(hd) == 64) return fa::Layout64::REQUEST;
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

extern "C" int fa_debug_force_path(int path) {
  if (path < 0 || path > 3) return FA_ERR_INVALID_ARG;
  fa::g_force_path.store(path);
  return FA_OK;
}

extern "C" int fa_debug_set_watchdog_ns(unsigned long long ns) {
  fa::g_watchdog_ns.store(ns == 0 ? fa::WATCHDOG_NS : ns);
  return FA_OK;
}
