// fa_persistent.cuh -- the persistent attention kernel (included by fa_prefill.cu).
//
// At most one CTA per SM walks a list of query-tile pairs ("units", numbered
// longest first as in the one-shot grid), or pieces of them, one after the
// other.  Per KV step it runs the one-shot kernel's chain unchanged (the pages'
// per-tile steps: minfer "53 · r50 — FA_TKV 32->16 occupancy experiment",
// section 2): TMA loads into a K/V ring, S = Q K^T and O += P V on the tensor
// core with accumulators in TMEM, a thread-per-row online softmax with a lazy
// O rescale.  What is new is how consecutive segments follow each other:
//
//   * one K/V ring and one sequence of (V_T, K_T+1) pair barriers run across
//     segment boundaries, so the next segment's first K tile streams in
//     behind the current segment's last V tile and the MMA thread waits once
//     per step, in and between segments alike;
//   * the next segment's Q is loaded right after its first K, once the last S
//     MMA of the segment that used the same buffer pair has read it (hd 128:
//     one Q buffer pair, loaded during the current segment's last step;
//     hd 64: two, a whole segment ahead), after an L2 prefetch;
//   * at hd 64, where TMEM has room for P beside S (as in fa_prefill64.cuh),
//     S_X(T+1) is issued as soon as softmax X has read S_X(T), not after
//     P V_X(T), so the tile's chain loses the MMA and its hand-offs;
//   * the softmax warps write a segment's output as soon as its last P V has
//     completed -- O / l rounded to 16 bits straight to the rows, or, for a
//     piece of a split unit, the unnormalised O with its m and l to the
//     workspace -- and go on to the next segment's first S tile, which the
//     tensor core has computed meanwhile.  (A fourth, epilogue warpgroup was
//     measured and removed: a 512-thread launch alone cost the step chain
//     ~5 %, more than the epilogue it took off the softmax warps.)
//
//   warps 0-3 / 4-7   softmax and epilogue of tile A / B (one thread per row == TMEM lane)
//   warp 8            MMA issuer (one thread; at hd 64 the whole warp, one lane issuing)
//   warp 9            TMA producer (one thread)
//   warps 10, 11      idle (they complete warpgroup 2)
//
// The work list comes in one of two forms.  Whole units (no workspace): CTA c
// takes units c, 2G-1-c, 2G+c, 4G-1-c, ... of the longest-first order (G CTAs,
// a snake, so long and short units pair up).  Stream-K ranges (a workspace):
// CTA c takes the contiguous range of (unit, KV step) work from (su[c], sj[c])
// to (su[c+1], sj[c+1]) of the split-KV schedule, and fa_sk_merge_kernel
// combines the split units' pieces afterwards.

namespace fa {

constexpr int PK_THREADS = NUM_THREADS;  // softmax A, softmax B, control
constexpr uint32_t PK_REGS_SOFTMAX = 208;
constexpr uint32_t PK_REGS_CONTROL = 56;
static_assert(128 * PK_REGS_CONTROL + 256 * PK_REGS_SOFTMAX <= NUM_THREADS * LAUNCH_REGS,
              "register split exceeds the launch allocation");

// Watchdog code of this kernel (bits 0-7 of g_fa_status), beside the shared ones.
enum : uint32_t {
  WD_SMEM_ALIGN = 17,  // the dynamic shared memory base is not 1024-byte aligned: nothing was run
};

template <int HD>
struct PkLayout {
  using L = Layout<HD>;
  static constexpr int NSLOT = HD == 128 ? 5 : 8;  // K/V ring depth
  static constexpr int NQB = HD == 128 ? 1 : 2;    // Q buffer pairs
  static constexpr int NPB = (NSLOT + 1) / 2;      // (V_T, K_T+1) pair barriers
  static constexpr int NPE = NSLOT / 2 + 1;        // hd 128: (K_T, V_T) pair-empty barriers
  static constexpr uint32_t QSET = 2 * L::Q_BYTES;  // Q_A, Q_B
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_RING = NQB * QSET;
  static constexpr uint32_t OFF_BAR = OFF_RING + NSLOT * L::SLOT_BYTES;
  // q_full[NQB], q_empty[NQB], pair[NPB], empty[NSLOT], s_full[2], p_full[2], o_full[2], drain,
  // s_free[2], pv_done[2] (hd 64: S and P in separate TMEM columns)
  static constexpr uint32_t NUM_BARS = 2 * NQB + NPB + NSLOT + 6 + 1 + 4;
  // TMEM: S_A | S_B | O_A | O_B, and at hd 64 P_A | P_B in the 128 columns left
  static constexpr uint32_t TM_P = L::TM_O + 2 * HD;
  static constexpr bool SPLIT_P = HD == 64;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;  // [0] TMEM base, [1] abort flag
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  // The kernel declares its dynamic shared memory 1024-byte aligned (the
  // 128-byte swizzle atoms need it) and checks the base, so no slack is asked.
  static constexpr uint32_t REQUEST = BYTES;
  static_assert(OFF_RING % 1024 == 0 && L::SLOT_BYTES % 1024 == 0, "swizzle atoms");
  static_assert(2 * NPB >= NSLOT && 2 * NPE > NSLOT && NPE <= NSLOT, "barrier reuse");
  static_assert(BYTES <= 232448, "shared memory per CTA");
};

struct PkParams {
  Params p;
  float4* ws_o;   // stream-K: partial O, float4 [piece slot][tile][HD/4][BM] (unused for whole units)
  float* ws_ml;   // stream-K: [piece slot][tile][2][BM]: m (log2 domain), l
  int ranges;     // 0: whole units in snake order over the grid; 1: stream-K ranges su / sj
  int n_units;
  int su[SK_MAX_CTAS + 1];  // stream-K: CTA c from (su[c], sj[c]) to (su[c+1], sj[c+1])
  int sj[SK_MAX_CTAS + 1];
  short pf[SK_MAX_CTAS];    // slot of CTA c's first segment when it continues a split unit, else -1
  short ph[SK_MAX_CTAS];    // slot of CTA c's last segment when it starts a split unit, else -1
};

// Segment k of CTA c: unit u, KV steps [jb, je).  False when the CTA has no
// segment k.  Every role walks the same sequence.
__device__ __forceinline__ bool pk_segment(const PkParams& sp, int c, int k, int& u, int& jb, int& je, UnitGeo& w) {
  if (!sp.ranges) {
    const int G = static_cast<int>(gridDim.x);
    u = (k & 1) ? (k + 1) * G - 1 - c : k * G + c;
    if (u >= sp.n_units) return false;
    w = unit_geo(sp.p, u);
    jb = 0;
    je = w.n;
    return true;
  }
  u = sp.su[c] + k;
  const int ue = sp.su[c + 1], je_last = sp.sj[c + 1];
  jb = k == 0 ? sp.sj[c] : 0;
  if (!(u < ue || (u == ue && jb < je_last))) return false;
  w = unit_geo(sp.p, u);
  je = u == ue ? je_last : w.n;
  return true;
}

template <int HD, bool BF16>
__global__ void __launch_bounds__(PK_THREADS, 1)
    fa_prefill_pk_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmKt,
                         const __grid_constant__ CUtensorMap tmVt, const __grid_constant__ PkParams sp) {
  const Params& p = sp.p;
  using L = Layout<HD>;
  using PL = PkLayout<HD>;
  constexpr int NSLOT = PL::NSLOT;
  constexpr int NQB = PL::NQB;
  constexpr int NPB = PL::NPB;
  constexpr int NPE = PL::NPE;
  constexpr bool PAIR_EMPTY = HD == 128;  // K_T and V_T freed on one commit (hd 64: per slot)
  extern __shared__ __align__(1024) uint8_t pk_smem[];
  const uint32_t sbase = ptx::smem_u32(pk_smem);
  if (sbase & 1023u) {  // uniform over the CTA: no barrier, TMEM or copy has been touched
    if (threadIdx.x == 0) atomicCAS(&g_fa_status, 0u, WD_SMEM_ALIGN);
    return;
  }
  const uint32_t sQ = sbase + PL::OFF_Q;
  const uint32_t sRing = sbase + PL::OFF_RING;
  const uint32_t bar = sbase + PL::OFF_BAR;
  auto bQfull = [&](int b) { return bar + 8u * b; };
  auto bQempty = [&](int b) { return bar + 8u * (NQB + b); };
  auto bPair = [&](int b) { return bar + 8u * (2 * NQB + b); };
  auto bEmpty = [&](int s) { return bar + 8u * (2 * NQB + NPB + s); };
  constexpr int B0 = 2 * NQB + NPB + NSLOT;
  auto bSfull = [&](int x) { return bar + 8u * (B0 + x); };
  auto bPfull = [&](int x) { return bar + 8u * (B0 + 2 + x); };
  auto bOfull = [&](int x) { return bar + 8u * (B0 + 4 + x); };
  const uint32_t bDrain = bar + 8u * (B0 + 6);
  auto bSfree = [&](int x) { return bar + 8u * (B0 + 7 + x); };   // hd 64: softmax X holds S_X in registers
  auto bPVdone = [&](int x) { return bar + 8u * (B0 + 9 + x); };  // hd 64: P V_X has read P_X, written O_X
  constexpr bool SPLIT_P = PL::SPLIT_P;
  static_assert(!SPLIT_P || PL::TM_P + 2 * (BN / 2) <= TMEM_COLS, "TMEM plan");
  uint32_t* misc = reinterpret_cast<uint32_t*>(pk_smem + PL::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = static_cast<int>(blockIdx.x);

  if (threadIdx.x == 0) {
    for (int b = 0; b < NQB; ++b) {
      ptx::mbar_init(bQfull(b), 1);
      ptx::mbar_init(bQempty(b), 1);
    }
    for (int b = 0; b < NPB; ++b) ptx::mbar_init(bPair(b), 2);  // one arrival per load of the pair
    for (int s = 0; s < NSLOT; ++s) ptx::mbar_init(bEmpty(s), 1);
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(bSfull(x), 1);
      ptx::mbar_init(bPfull(x), BM);   // every softmax thread of the tile
      ptx::mbar_init(bOfull(x), 1);
      ptx::mbar_init(bSfree(x), BM);  // every softmax thread of the tile
      ptx::mbar_init(bPVdone(x), 1);
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
  // set-up overlaps the previous kernel in the stream; global memory only after it
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();

  if (warp >= MMA_WARP) {
    ptx::setmaxnreg_dec<PK_REGS_CONTROL>();
    if (warp == PRODUCER_WARP && lane == 0) {
      // ------------------------------------------------------------ producer
      // Loads in one sequence over all segments: K_T at g = 2T, V_T at
      // g = 2T + 1 (T counts KV steps over the CTA's segments), load g in ring
      // slot g % NSLOT.  K_0 completes on the first Q barrier; V_T and K_T+1 on
      // pair barrier T % NPB, whichever segments they belong to.  Segment s's
      // Q is loaded before its first K (once the Q buffer pair it reuses is
      // free).
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      if (p.block_table) {
        ptx::prefetch_tmap(&tmKt);
        ptx::prefetch_tmap(&tmVt);
      }
      int g = 0, nq = 0;
      bool ok = true;
      int u = 0, jb = 0, je = 0;
      UnitGeo w{};
      // Q of the segment into its buffer pair, once the pair is free (the last
      // S MMA of the segment NQB earlier has read it); the first segment's Q
      // completes on the same barrier as K_0
      auto load_q = [&](int k) -> bool {
        const int qb = nq % NQB;
        if (nq >= NQB && !wait_bar(bQempty(qb), ((nq - NQB) / NQB) & 1, abort_flag, p.watchdog_ns, WD_PRODUCER_EMPTY))
          return false;
        ptx::mbar_arrive_expect_tx(bQfull(qb), L::Q_BYTES * (w.has1 ? 2u : 1u) + (g == 0 ? L::SLOT_BYTES : 0u));
        const uint32_t dq = sQ + qb * PL::QSET;
#pragma unroll
        for (int c = 0; c < (int)L::KCH; ++c)
          ptx::tma_load_4d(dq + c * (BM * 128), &tmQ, bQfull(qb), c * 64, w.hq0, w.q00, w.b);
        if (w.has1) {
#pragma unroll
          for (int c = 0; c < (int)L::KCH; ++c)
            ptx::tma_load_4d(dq + L::Q_BYTES + c * (BM * 128), &tmQ, bQfull(qb), c * 64, w.hq1, w.q01, w.b);
        }
        ++nq;
        int u2, jb2, je2;  // warm L2 with the next segment's Q
        UnitGeo w2;
        if (pk_segment(sp, cta, k + 1, u2, jb2, je2, w2)) {
#pragma unroll
          for (int c = 0; c < (int)L::KCH; ++c) {
            ptx::tma_prefetch_l2_4d(&tmQ, c * 64, w2.hq0, w2.q00, w2.b);
            if (w2.has1) ptx::tma_prefetch_l2_4d(&tmQ, c * 64, w2.hq1, w2.q01, w2.b);
          }
        }
        return true;
      };
      for (int k = 0; ok && pk_segment(sp, cta, k, u, jb, je, w); ++k) {
        if (je <= jb) continue;  // nothing to stream (the epilogue writes zeros)
        // The CTA's first Q goes before K_0.  A later segment's Q goes after
        // its first K: that K completes the previous segment's last pair
        // barrier, which must not wait for the Q buffer to free up.
        if (g == 0) ok = load_q(k);
        if (!ok) break;
        int page = -1, blk = 0;  // paged K/V: the pool block of the current page
        for (int i = 2 * jb; i < 2 * je; ++i, ++g) {
          const int s = g % NSLOT;
          if (g >= NSLOT) {
            if constexpr (PAIR_EMPTY) {  // the previous occupant, load g - NSLOT, belongs to step e
              const int e = (g - NSLOT) >> 1;
              ok = wait_bar(bEmpty(e % NPE), (e / NPE) & 1, abort_flag, p.watchdog_ns, WD_PRODUCER_EMPTY);
            } else {
              ok = wait_bar(bEmpty(s), ((g / NSLOT) & 1) ^ 1u, abort_flag, p.watchdog_ns, WD_PRODUCER_EMPTY);
            }
          }
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
                atomicCAS(&g_fa_status, 0u, WD_PAGE_BLOCK | ((blockIdx.x < 0xFFFFFFu ? blockIdx.x : 0xFFFFFFu) << 8));
                blk = p.num_blocks;
              }
            }
            row = key0 - pg * p.page_size;
            bat = blk;
            tail = pg == p.last_page;
          }
          const int pj = (g - 1) >> 1;  // pair of load g (V_pj, K_pj+1)
          const uint32_t fb = g == 0 ? bQfull(0) : bPair(pj % NPB);
          // pair pj reuses pair pj-NPB's barrier: that phase must have completed
          if ((g & 1) && pj >= NPB) ok = wait_bar(fb, ((pj - NPB) / NPB) & 1, abort_flag, p.watchdog_ns, WD_PRODUCER_EMPTY);
          if (!ok) break;
          if (g > 0) ptx::mbar_arrive_expect_tx(fb, L::SLOT_BYTES);
          const CUtensorMap* m = (i & 1) ? (tail ? &tmVt : &tmV) : (tail ? &tmKt : &tmK);
#pragma unroll
          for (int c = 0; c < (int)L::KCH; ++c)
            ptx::tma_load_4d(sRing + s * L::SLOT_BYTES + c * (BN * 128), m, fb, c * 64, w.hk, row, bat);
          if (i == 2 * jb && g > 0) {  // (g > 0: the Q barrier expects no K bytes)
            ok = load_q(k);
            if (!ok) break;
          }
        }
      }
      // the last pair has no K (or a CTA gave up after a V): its second arrival without bytes
      if (g >= 2 && (g & 1) == 0) ptx::mbar_arrive(bPair(((g - 2) >> 1) % NPB));
      // every copy issued has landed before the CTA exits
      for (int b = 0; b < NQB && b < nq; ++b) {
        const int last = b + NQB * ((nq - 1 - b) / NQB);
        drain_wait(bQfull(b), (last / NQB) & 1, DRAIN_NS);
      }
      const int npairs = g / 2;
      for (int b = 0; b < NPB && b < npairs; ++b) {
        const int last = b + NPB * ((npairs - 1 - b) / NPB);
        drain_wait(bPair(b), (last / NPB) & 1, DRAIN_NS);
      }
    } else if (warp == MMA_WARP && (HD == 64 || lane == 0)) {
      // hd 64: the whole warp runs the loop and the waits, one elected lane
      // issues (as in the one-shot kernel); hd 128: lane 0 alone
      constexpr bool CONV = HD == 64;
      const bool leader = CONV ? ptx::elect_one() : true;
      // ---------------------------------------------------------- MMA issuer
      // Per segment: S_A(T0), S_B(T0) with K_T0, then per step T the one-shot
      // order P V_A(T), S_A(T+1), P V_B(T), S_B(T+1) -- at hd 64, where P has
      // columns of its own, S_X(T+1) goes first, as soon as softmax X has read
      // S_X(T).  The first P V of a tile in a segment overwrites its O; it
      // waits for that tile's first P, which the softmax writes only after it
      // has read the previous segment's O.  The segment's first S overwrites
      // S_X: its softmax read the last S before writing the last P.
      constexpr uint32_t IDESC_S = ptx::idesc_f16(BF16, BM, BN, false, false);  // Q, K both K-major
      constexpr uint32_t IDESC_O = ptx::idesc_f16(BF16, BM, HD, false, true);   // P from TMEM, V MN-major
      constexpr uint32_t DHI = ptx::sdesc_sw128_hi(1024);
      // The descriptor bases pass through an opaque move at hd 128, where
      // without it the compiler hoists them into registers the MMA thread
      // does not have (spills); at hd 64 they need no help (measured +1 to +2 %).
      auto launder = [](uint32_t v) { return HD == 64 ? v : ptx::opaque(v); };
      auto issue_s = [&](int x, uint32_t qset, int slot) {
        const uint32_t d = tmem + L::TM_S + x * BN;
        const uint32_t q = launder(ptx::sdesc_sw128_lo(qset + x * L::Q_BYTES, 16));
        const uint32_t kd = launder(ptx::sdesc_sw128_lo(sRing + slot * L::SLOT_BYTES, 16));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t o = ((kk / 4) * (BM * 128) + (kk % 4) * 32) >> 4;
          if (leader) ptx::mma_f16_ss(d, ptx::sdesc_join(q + o, DHI), ptx::sdesc_join(kd + o, DHI), IDESC_S, kk > 0 ? 1u : 0u);
        }
        if (leader) ptx::mma_commit(bSfull(x));
      };
      auto issue_pv = [&](int x, int slot, bool acc) {
        const uint32_t d = launder(tmem + L::TM_O + x * HD);
        // P_X, 2 elements per column: over S_X (hd 128) or in its own columns (hd 64)
        const uint32_t a = launder(tmem + (SPLIT_P ? PL::TM_P + x * (BN / 2) : L::TM_S + x * BN));
        const uint32_t v = launder(ptx::sdesc_sw128_lo(sRing + slot * L::SLOT_BYTES, BN * 128));
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          if (leader) ptx::mma_f16_ts(d, a + kk * 8, ptx::sdesc_join(v + kk * ((16 * 128) >> 4), DHI), IDESC_O,
                          (acc || kk > 0) ? 1u : 0u);
        if constexpr (SPLIT_P) {
          if (leader) ptx::mma_commit(bPVdone(x));
        }
      };
      int T = 0;               // KV steps issued over the CTA's segments
      int pc0 = 0, pc1 = 0;    // tiles of A / B so far (s_full / p_full phases)
      int nq = 0;
      bool ok = true;
      int u = 0, jb = 0, je = 0;
      UnitGeo w{};
      for (int k = 0; ok && pk_segment(sp, cta, k, u, jb, je, w); ++k) {
        if (je <= jb) continue;
        const int nseg = je - jb;
        const int nAs = max(0, min(je, w.nA) - jb);
        const int nBs = max(0, min(je, w.nB) - jb);
        const int qb = nq % NQB;
        ok = mma_wait<CONV>(bQfull(qb), (nq / NQB) & 1, abort_flag, p.watchdog_ns, WD_MMA_Q);  // Q (and K_0)
        if (!ok) break;
        const uint32_t qset = sQ + qb * PL::QSET;
        ptx::tc_fence_after();
        const int sk0 = (2 * T) % NSLOT;  // K_T (arrived with Q, or with the pair of the previous step)
        if (nAs > 0) issue_s(0, qset, sk0);
        if (nBs > 0) issue_s(1, qset, sk0);
        if constexpr (!PAIR_EMPTY) {
          if (leader) ptx::mma_commit(bEmpty(sk0));
        }
        if (NQB == 1 && nseg == 1 && leader) ptx::mma_commit(bQempty(qb));
        for (int t = 0; t < nseg; ++t, ++T) {
          const int sv = (2 * T + 1) % NSLOT;  // V_T
          const int sk = (2 * T + 2) % NSLOT;  // K_T+1
          ok = mma_wait<CONV>(bPair(T % NPB), (T / NPB) & 1, abort_flag, p.watchdog_ns, WD_MMA_KV_FULL);
          if (!ok) break;
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            const int nXs = x == 0 ? nAs : nBs;
            if (t < nXs) {
              const int tile = (x == 0 ? pc0 : pc1) + t;  // tiles of X so far (barrier phases)
              if constexpr (SPLIT_P) {  // S_X(T+1) as soon as softmax X holds S_X(T) in registers
                if (t + 1 < nXs) {
                  ok = mma_wait<CONV>(bSfree(x), tile & 1, abort_flag, p.watchdog_ns, WD_MMA_S_FREE);
                  if (!ok) break;
                  ptx::tc_fence_after();
                  issue_s(x, qset, sk);
                }
              }
              ok = mma_wait<CONV>(bPfull(x), tile & 1, abort_flag, p.watchdog_ns, WD_MMA_P_FULL);
              if (!ok) break;
              ptx::tc_fence_after();
              issue_pv(x, sv, t > 0);
            }
            if constexpr (PAIR_EMPTY) {
              if (x == 1 && leader) ptx::mma_commit(bEmpty(T % NPE));  // K_T (its S MMAs came earlier) and V_T
            }
            if (!SPLIT_P && t + 1 < nXs) issue_s(x, qset, sk);
          }
          if (!ok) break;
          if constexpr (!PAIR_EMPTY) {
            // V_T: both tiles' P V(T) are issued (committed after the tile loop, as
            // in the one-shot kernel: measured ~1 % faster at hd 64 than inside it)
            if (leader) ptx::mma_commit(bEmpty(sv));
            if (t + 1 < nseg && leader) ptx::mma_commit(bEmpty(sk));
          }
          if constexpr (NQB == 1) {
            if (t + 2 == nseg && leader) ptx::mma_commit(bQempty(qb));  // the segment's last S MMAs are issued
          }
        }
        if (!ok) break;
        // two Q buffers (hd 64): released with the segment, a commit out of the
        // step loop (the loop's per-step test cost ~2 % at hd 64)
        if (NQB > 1 && leader) ptx::mma_commit(bQempty(qb));
        if (nAs > 0 && leader) ptx::mma_commit(bOfull(0));
        if (nBs > 0 && leader) ptx::mma_commit(bOfull(1));
        pc0 += nAs;
        pc1 += nBs;
        ++nq;
      }
      // every MMA issued has finished before TMEM is freed
      if (leader) ptx::mma_commit(bDrain);
      drain_wait(bDrain, 0, DRAIN_NS);
    }
  } else {
    ptx::setmaxnreg_inc<PK_REGS_SOFTMAX>();
    // -------------------------------------------------------------- softmax
    const int x = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + L::TM_S + x * BN;
    const uint32_t tO = tmem + lane_off + L::TM_O + x * HD;
    const uint32_t tP = SPLIT_P ? tmem + lane_off + PL::TM_P + x * (BN / 2) : tS;  // P_X
    const int off = p.Skv - p.Sq;
    const float sl2 = p.sl2;
    int cnt = 0;   // tiles processed (s_full / p_full phases)
    int ocnt = 0;  // segments with tiles of x (o_full phases)
    // O / l of row r rounded to 16 bits, straight to the output row (32-byte
    // stores where the row is 32-byte aligned), up to the head's true width;
    // and the row's log-sum-exp when asked for
    auto store_row = [&](int q0, int hq, int b, float m, float l, const uint32_t (&orr)[HD]) {
      if (q0 + r >= p.Sq) return;
      if (p.lse) p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.Sq + q0 + r] = row_lse(m, l);
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      uint16_t* orow = p.o + ((static_cast<size_t>(b) * p.Sq + q0 + r) * p.Hq + hq) * p.hd;
      const bool a32 = (reinterpret_cast<uintptr_t>(orow) & 31u) == 0;
#pragma unroll
      for (int c = 0; c < HD / 16; ++c) {
        if (16 * c >= p.hd) break;
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          pk[e] = pack2<BF16>(__uint_as_float(orr[16 * c + 2 * e]) * inv_l, __uint_as_float(orr[16 * c + 2 * e + 1]) * inv_l);
        if (a32 && 16 * c + 16 <= p.hd) {
          ptx::st_global_v8(orow + 16 * c, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
        } else {
          *reinterpret_cast<uint4*>(orow + 16 * c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          if (16 * c + 8 < p.hd) *reinterpret_cast<uint4*>(orow + 16 * c + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
    };
    bool ok = true;
    int u = 0, jb = 0, je = 0;
    UnitGeo w{};
    for (int k = 0; ok && pk_segment(sp, cta, k, u, jb, je, w); ++k) {
      const int q0 = x == 0 ? w.q00 : w.q01;
      const int nX = x == 0 ? w.nA : w.nB;
      const int jx_end = min(je, nX);
      const int hqx = x == 0 ? w.hq0 : w.hq1;
      if (jx_end <= jb) {  // no KV tile of x in this segment
        if (x == 1 && !w.has1) continue;
        if (jb == 0 && je >= w.n) {  // a whole unit whose rows see no key: O = 0
          uint32_t orr[HD];
#pragma unroll
          for (int e = 0; e < HD; ++e) orr[e] = 0u;
          store_row(q0, hqx, w.b, -INFINITY, 0.f, orr);
        } else {
          const int ps = jb == 0 ? sp.ph[cta] : sp.pf[cta];
          if (ps >= 0) {
            const size_t slot_t = static_cast<size_t>(ps) * 2 + x;
            sp.ws_ml[(slot_t * 2 + 0) * BM + r] = -INFINITY;
            sp.ws_ml[(slot_t * 2 + 1) * BM + r] = 0.f;
          }
        }
        continue;
      }
      const int kv_all = p.causal ? min(p.Skv, off + q0 + 1) : p.Skv;       // keys every row sees
      const int row_lim = p.causal ? min(p.Skv, off + q0 + r + 1) : p.Skv;  // keys this row sees
      float m_ref = -INFINITY;  // running max (log2 domain) that O and l are scaled to
      float l = 0.f;
      for (int j = jb; j < jx_end; ++j, ++cnt) {
        ok = warp_wait_bar(bSfull(x), cnt & 1, abort_flag, p.watchdog_ns, WD_SOFTMAX_S_FULL);
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t sr[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) ptx::tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
        ptx::tmem_wait_ld();
        ptx::reg_fence(sr);
        if constexpr (SPLIT_P) {  // S_X is in registers: the tensor core may compute S_X(T+1) over it
          ptx::tc_fence_before();
          ptx::mbar_arrive(bSfree(x));
        }
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
        float mk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mk[e] = ptx::fmax3(s[e], s[8 + e], s[16 + e]);
#pragma unroll
        for (int t = 3; t < 15; t += 2)
#pragma unroll
          for (int e = 0; e < 8; ++e) mk[e] = ptx::fmax3(mk[e], s[8 * t + e], s[8 * t + 8 + e]);
#pragma unroll
        for (int e = 0; e < 8; ++e) mk[e] = fmaxf(mk[e], s[120 + e]);
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
        // the running max moved: rescale O_X in TMEM (hd 128: P V_X(j-1) finished
        // before S_X(j) did; hd 64: waited for above)
        if constexpr (SPLIT_P) {
          // P V_X of the previous tile of this segment has read P_X and written
          // O_X before this tile touches either (at a segment's first tile the
          // o_full wait of the previous segment covered it)
          if (j > jb) {
            ok = warp_wait_bar(bPVdone(x), (cnt - 1) & 1, abort_flag, p.watchdog_ns, WD_SOFTMAX_PV_DONE);
            if (!ok) break;
            ptx::tc_fence_after();
          }
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
        // P_X over the first BN/2 columns of S_X (hd 128) or into its own (hd 64)
        ptx::tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&pp[0]));
        ptx::tmem_st32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&pp[32]));
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bPfull(x));
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue
      // O_X of this segment is final once its last P V has completed; it is
      // read out before this thread writes the next segment's first P, which
      // is what lets the MMA thread overwrite O_X.
      ok = warp_wait_bar(bOfull(x), ocnt & 1, abort_flag, p.watchdog_ns, WD_SOFTMAX_O_DONE);
      if (!ok) break;
      ++ocnt;
      ptx::tc_fence_after();
      uint32_t orr[HD];  // the whole row: all loads in flight before one wait
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) ptx::tmem_ld32(tO + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&orr[c * 32]));
      ptx::tmem_wait_ld();
      ptx::reg_fence(orr);
      if (jb == 0 && je >= w.n) {  // a whole unit: O / l to the row
        store_row(q0, hqx, w.b, m_ref, l, orr);
      } else {  // a piece of a split unit: (O, m, l) to its workspace slot
        const int ps = jb == 0 ? sp.ph[cta] : sp.pf[cta];
        if (ps < 0) {
          if (lane == 0) atomicCAS(&g_fa_status, 0u, WD_PIECE_SLOT | ((blockIdx.x < 0xFFFFFFu ? blockIdx.x : 0xFFFFFFu) << 8));
          continue;
        }
        const size_t slot_t = static_cast<size_t>(ps) * 2 + x;
        float4* dst = sp.ws_o + slot_t * (HD / 4) * BM + r;
#pragma unroll
        for (int e = 0; e < HD / 4; ++e)
          dst[e * BM] = make_float4(__uint_as_float(orr[4 * e]), __uint_as_float(orr[4 * e + 1]),
                                    __uint_as_float(orr[4 * e + 2]), __uint_as_float(orr[4 * e + 3]));
        sp.ws_ml[(slot_t * 2 + 0) * BM + r] = m_ref;
        sp.ws_ml[(slot_t * 2 + 1) * BM + r] = l;
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
