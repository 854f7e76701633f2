// fa_prefill_pair.cuh -- the one-shot kernel on CTA pairs, for heads 72 to 128
// wide and GQA groups of a multiple of 4 query heads (included by
// fa_prefill.cu).
//
// The per-tile steps are the pages' (minfer "53 · r50 — FA_TKV 32->16
// occupancy experiment", section 2: S = Q K^T, mask, max, exp, sum, rescale O,
// O += P V), on Blackwell's paired MMAs: a cluster of two CTAs on two SMs,
// whose MMAs (tcgen05 cta_group::2, M = 256) take rows 0-127 of a 256-row tile
// from CTA 0 and rows 128-255 from CTA 1, and split the B operand along N, so
// that each CTA loads only half of every K and V tile.
//
// A pair owns four query heads of one KV head at the same 128 rows: CTA r has
// heads 4g + r (tile A) and 4g + 2 + r (tile B).  The paired tile A is heads
// 4g, 4g + 1; the paired tile B heads 4g + 2, 4g + 3; all four read the same
// K/V tiles.  Per CTA and KV tile j: keys [128 j + 64 r, +64) of K (all of hd)
// and columns [64 r, +64) of V (all 128 keys), 16 KB each.
//
// What the halved operand traffic buys: P lives in shared memory (each CTA
// its own 128 rows, the A operand of P V), not over S in TMEM.  So S_X(j+1)
// is issued as soon as both CTAs' softmax X have read S_X(j) (an s_free
// barrier), before P V_X(j): the tensor core computes the next S while the
// softmax works on this one, and the MMAs and their hand-offs drop out of a
// tile's chain.  Softmax X waits for P V_X(j-1) (pv_done) before it rescales
// O_X or writes P_X(j).  (With P also in shared memory, one CTA alone would
// need more shared-memory bandwidth than an SM has.)
//
//   TMEM (512 columns, allocated jointly): S_A | S_B | O_A | O_B, 128 each
//   shared memory per CTA: Q_A, Q_B, P_A, P_B (32 KB each), a ring of six
//     16 KB K/V halves, barriers
//
//   warp 9 (both CTAs)   TMA producer: Q_A, Q_B, then the K/V halves, each
//                        load counted on its own CTA's barriers (which it
//                        drains before exit)
//   warp 11 (both CTAs)  forwards its CTA's load completions to CTA 0's joint
//                        barriers, which the MMA issuers wait on
//   warps 8, 10 (CTA 0)  the MMA issuers of tiles A and B for both CTAs, each
//                        in its tile's own order (S_X(j+1) after s_free,
//                        P V_X(j) after p_full); their commits arrive on the
//                        barrier of the same address in both CTAs, and the
//                        ring slots, o_final and the drain count one commit
//                        per issuer
//   warps 0-7 (both)     softmax of tiles A (0-3) and B (4-7), one thread per
//                        row == TMEM lane; their s_free and p_full arrivals go
//                        to CTA 0's barriers
//
// CTA 1's p_full arrivals and forwarded load completions publish shared
// memory that CTA 0's MMAs read: they release at cluster scope, and CTA 0
// waits with acquire at cluster scope.  Its s_free arrivals publish nothing
// (S is in registers by then) and are plain signals.
//
// Measured (8192-token GQA prefill): slower than the single-CTA kernel (see
// the library's path selection), so this kernel runs only when asked for.
// The softmax of a tile takes longer here (the P stores, the proxy fence,
// the cross-CTA arrivals), and the two tiles' softmax warps, which share the
// SM's four schedulers, end up running in phase.
//
// Every wait is bounded as in the other kernels.  Before either CTA frees the
// joint TMEM or exits, both pass a cluster barrier: the MMAs of CTA 0 read
// CTA 1's shared memory, and CTA 1's threads arrive on CTA 0's barriers.

namespace fa {

// Watchdog codes of this kernel (bits 0-7 of g_fa_status), beside the shared ones.
enum : uint32_t {
  WD_PAIR_FORWARD = 13,  // a forwarder waiting for its own CTA's loads
};

// Register split: the MMA thread builds two operand addresses per MMA (Q or
// P, and a K or V half) and spills at 56; the whole launch allocation is used.
constexpr uint32_t PAIR_REGS_CONTROL = 88;
static_assert(128 * PAIR_REGS_CONTROL + 256 * REGS_SOFTMAX <= NUM_THREADS * LAUNCH_REGS,
              "register split exceeds the launch allocation");

struct PairLayout {
  static constexpr int HD = 128;
  static constexpr uint32_t Q_BYTES = BM * HD * 2;       // one query tile (32 KB)
  static constexpr uint32_t P_BYTES = BM * BN * 2;       // one P tile (32 KB)
  static constexpr uint32_t HALF_BYTES = 64 * HD * 2;    // half a K tile == half a V tile (16 KB)
  static constexpr int NSLOT = 6;                        // K/V ring depth, in halves
  static constexpr int NPB = 3;                          // (V_j, K_j+1) pair barriers
  static constexpr uint32_t OFF_Q = 0;                   // Q_A, Q_B
  static constexpr uint32_t OFF_P = 2 * Q_BYTES;         // P_A, P_B (and the O staging at the end)
  static constexpr uint32_t OFF_RING = OFF_P + 2 * P_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_RING + NSLOT * HALF_BYTES;
  // q_full, pair[NPB] (this CTA's own loads), empty[NSLOT], s_full[2], s_free[2],
  // p_full[2], pv_done[2], o_final, drain, o_staged[2], jq_full, jpair[NPB] (both
  // CTAs' loads, used in CTA 0)
  static constexpr uint32_t NUM_BARS = 1 + NPB + NSLOT + 2 + 2 + 2 + 2 + 1 + 1 + 2 + 1 + NPB;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;  // [0] TMEM base, [1] abort flag
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static constexpr uint32_t REQUEST = BYTES + 1024;  // slack to align the dynamic base
  static constexpr uint32_t TM_S = 0;                // S_A, S_B
  static constexpr uint32_t TM_O = 2 * BN;           // O_A, O_B
  static_assert(TM_O + 2 * HD <= TMEM_COLS, "TMEM plan");
  static_assert(OFF_P % 1024 == 0 && OFF_RING % 1024 == 0 && HALF_BYTES % 1024 == 0, "swizzle atoms");
  static_assert(NSLOT % 2 == 0 && 2 * NPB == NSLOT, "pair j and pair j + NPB use the same two slots");
  static_assert(REQUEST <= 232448, "shared memory per CTA");
};

// The pair's unit: longest query tiles first; the clusters of one KV head's
// quads are adjacent, so their K/V tiles come from L2.
struct PairWork {
  int b, hk, q0;
  int hq[2];  // this CTA's heads: tile A, tile B
};

__device__ __forceinline__ PairWork decode_pair_work(const Params& p, int unit, uint32_t rank) {
  const int quads = p.Hq / 4;
  const int per_qt = quads * p.B;
  const int qt = p.n_qtiles - 1 - unit / per_qt;
  const int rem = unit % per_qt;
  PairWork w;
  w.b = rem / quads;
  const int g = rem % quads;
  w.hq[0] = 4 * g + static_cast<int>(rank);
  w.hq[1] = 4 * g + 2 + static_cast<int>(rank);
  w.hk = (4 * g) / p.G;
  w.q0 = qt * BM;
  return w;
}

// Bounded waits on barriers that the other CTA arrives on (acquire at
// cluster scope); otherwise as wait_bar / warp_wait_bar.
__device__ __forceinline__ bool wait_bar_cl(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                            unsigned long long limit_ns, uint32_t code) {
  if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  const bool fine = limit_ns < 1000000ull;
  while (true) {
#pragma unroll 1
    for (int i = 0; i < (fine ? 1 : 32); ++i)
      if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > limit_ns) {
      give_up_wait(abort_flag, code);
      return false;
    }
  }
}

// The arrival of one warp (lane 0, after the warp's own writes) on CTA 0's
// barrier: with a cluster-scope release when it publishes shared memory the
// other CTA's MMAs read (P), else as a plain signal (S read into registers).
template <bool kPublishes>
__device__ __forceinline__ void warp_arrive_leader(uint32_t bar, uint32_t rank, int lane) {
  __syncwarp();
  if (lane == 0) {
    if (rank == 0) ptx::mbar_arrive(bar);
    else if (kPublishes) ptx::mbar_arrive_cluster(ptx::mapa(bar, 0));
    else ptx::mbar_arrive_remote_signal(ptx::mapa(bar, 0));
  }
}

template <bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    fa_prefill_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKh,
                           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                           const Params p) {
  constexpr int HD = 128;
  using L = PairLayout;
  constexpr int NSLOT = L::NSLOT;
  constexpr int NPB = L::NPB;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;  // the same in both CTAs: the descriptors name one address
  uint8_t* gbase = smem_raw + (sbase - raw);

  const uint32_t sQ = sbase + L::OFF_Q;
  const uint32_t sP = sbase + L::OFF_P;
  const uint32_t sRing = sbase + L::OFF_RING;
  const uint32_t bar = sbase + L::OFF_BAR;
  const uint32_t bQ = bar;
  auto bPair = [&](int b) { return bar + 8u * (1 + b); };  // b < NPB
  auto bEmpty = [&](int s) { return bar + 8u * (1 + NPB + s); };
  constexpr int B0 = 1 + NPB + NSLOT;
  auto bSfull = [&](int x) { return bar + 8u * (B0 + x); };
  auto bSfree = [&](int x) { return bar + 8u * (B0 + 2 + x); };
  auto bPfull = [&](int x) { return bar + 8u * (B0 + 4 + x); };
  auto bPVdone = [&](int x) { return bar + 8u * (B0 + 6 + x); };
  const uint32_t bOfinal = bar + 8u * (B0 + 8);
  const uint32_t bDrain = bar + 8u * (B0 + 9);
  auto bOstaged = [&](int x) { return bar + 8u * (B0 + 10 + x); };
  const uint32_t bJQ = bar + 8u * (B0 + 12);                        // CTA 0: both CTAs' Q and K_0
  auto bJPair = [&](int b) { return bar + 8u * (B0 + 13 + b); };  // CTA 0: both CTAs' pair b
  uint32_t* misc = reinterpret_cast<uint32_t*>(gbase + L::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_rank();
  const PairWork w = decode_pair_work(p, static_cast<int>(blockIdx.x >> 1), rank);
  const int n = kv_tiles(p, w.q0, true);  // KV tiles of the unit (the same for all four heads)

  if (threadIdx.x == 0) {
    // q_full and pair count this CTA's own loads (its producer drains on
    // them); CTA 0's jq_full and jpair count one forwarded completion from
    // each CTA, and its s_free and p_full one arrival per softmax warp of
    // both CTAs
    ptx::mbar_init(bQ, 1);
    for (int b = 0; b < NPB; ++b) {
      ptx::mbar_init(bPair(b), 2);
      ptx::mbar_init(bJPair(b), 2);
    }
    ptx::mbar_init(bJQ, 2);
    for (int s = 0; s < NSLOT; ++s) ptx::mbar_init(bEmpty(s), 2);  // one commit per MMA issuer
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(bSfull(x), 1);
      ptx::mbar_init(bSfree(x), 8);
      ptx::mbar_init(bPfull(x), 8);
      ptx::mbar_init(bPVdone(x), 1);
      ptx::mbar_init(bOstaged(x), 4);  // one arrival per softmax warp of the tile
    }
    ptx::mbar_init(bOfinal, 2);
    ptx::mbar_init(bDrain, 2);
    misc[1] = 0u;
    ptx::mbar_fence_init();
  }
  if (warp == MMA_WARP) {
    ptx::tmem_alloc_pair(ptx::smem_u32(misc), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers exist before either CTA arrives on the other's
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();

  if (warp >= MMA_WARP) {
  ptx::setmaxnreg_dec<PAIR_REGS_CONTROL>();
  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    // Q_A, Q_B and K_0 on the Q barrier, then V_j and K_j+1 on pair barrier
    // j % NPB; load i in slot i % NSLOT, each slot freed by its own commit.
    // This CTA's halves: K rows 128 j + 64 rank, V columns 64 rank.
    if (lane == 0) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmKh);
      ptx::prefetch_tmap(&tmV);
      ptx::prefetch_tmap(&tmO);
      const int kr = 64 * static_cast<int>(rank);
      ptx::mbar_arrive_expect_tx(bQ, 2 * L::Q_BYTES + (n > 0 ? L::HALF_BYTES : 0u));
      for (int x = 0; x < 2; ++x) {
        ptx::tma_load_4d(sQ + x * L::Q_BYTES, &tmQ, bQ, 0, w.hq[x], w.q0, w.b);
        ptx::tma_load_4d(sQ + x * L::Q_BYTES + BM * 128, &tmQ, bQ, 64, w.hq[x], w.q0, w.b);
      }
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < 2 * n; ++i) {
        const int s = i % NSLOT;
        if (i >= NSLOT) ok = wait_bar(bEmpty(s), ((i / NSLOT) & 1) ^ 1u, abort_flag, p.watchdog_ns, WD_PRODUCER_EMPTY);
        if (!ok) break;
        const int pj = (i - 1) >> 1;  // pair of load i (V_pj, K_pj+1)
        const uint32_t fb = i == 0 ? bQ : bPair(pj % NPB);
        // pair pj reuses pair pj-NPB's barrier: that phase must have completed
        if ((i & 1) && pj >= NPB) ok = wait_bar(fb, ((pj - NPB) / NPB) & 1, abort_flag, p.watchdog_ns, WD_PRODUCER_EMPTY);
        if (!ok) break;
        if (i > 0) ptx::mbar_arrive_expect_tx(fb, L::HALF_BYTES);
        const uint32_t dst = sRing + s * L::HALF_BYTES;
        const int key0 = (i >> 1) * BN;
        if (i & 1) {  // V_j: all keys, this CTA's 64 columns
          ptx::tma_load_4d(dst, &tmV, fb, kr, w.hk, key0, w.b);
        } else {      // K_j: this CTA's 64 keys, both 64-column blocks of hd
          ptx::tma_load_4d(dst, &tmKh, fb, 0, w.hk, key0 + kr, w.b);
          ptx::tma_load_4d(dst + 64 * 128, &tmKh, fb, 64, w.hk, key0 + kr, w.b);
        }
        ++issued;
      }
      // a pair whose K was not issued (the last V, or a CTA that gave up):
      // its second arrival without bytes
      if (issued >= 2 && (issued & 1) == 0) ptx::mbar_arrive(bPair(((issued - 2) >> 1) % NPB));
      // every copy issued has landed before the CTA exits
      drain_wait(bQ, 0, DRAIN_NS);
      const int npairs = issued / 2;  // pairs armed
      for (int b = 0; b < NPB && b < npairs; ++b) {
        const int last = b + NPB * ((npairs - 1 - b) / NPB);
        drain_wait(bPair(b), (last / NPB) & 1, DRAIN_NS);
      }
    }
  } else if (warp == PRODUCER_WARP + 2) {
    // ----------------------------------------------------------- forwarder
    // A CTA's own load barriers complete when its halves have landed; each
    // completion becomes one arrival on CTA 0's joint barrier (a cluster
    // release from CTA 1: its shared memory is what CTA 0's MMAs read).
    // (Pair j + NPB of a CTA cannot complete before pair j was forwarded: its
    // loads reuse the slots of pair j, which CTA 0's MMAs free only after
    // they waited for the joint pair j.)
    if (lane == 0) {
      auto forward = [&](uint32_t jb) {
        if (rank == 0) ptx::mbar_arrive(jb);
        else ptx::mbar_arrive_cluster(ptx::mapa(jb, 0));
      };
      // (the Q barrier always: CTA 0 waits for it even when the unit has no KV tile)
      bool ok = wait_bar(bQ, 0, abort_flag, p.watchdog_ns, WD_PAIR_FORWARD);
      if (ok) forward(bJQ);
      for (int j = 0; ok && j < n; ++j) {
        ok = wait_bar(bPair(j % NPB), (j / NPB) & 1, abort_flag, p.watchdog_ns, WD_PAIR_FORWARD);
        if (ok) forward(bJPair(j % NPB));
      }
    }
  } else if ((warp == MMA_WARP || warp == PRODUCER_WARP + 1) && rank == 0 && lane == 0) {
    const int xi = warp == MMA_WARP ? 0 : 1;  // the tile this thread issues for
    // ---------------------------------------------------------- MMA issuers
    // Issuer X, per KV step j: S_X(j+1) once both softmax X hold S_X(j) in
    // registers, then P V_X(j) once both have written P_X(j).  (One issuer
    // for both tiles, in either fixed order, measured 7 to 20 % slower: a
    // wait for one tile's P holds back the other tile's next S.)
    constexpr uint32_t IDESC_S = ptx::idesc_f16(BF16, 2 * BM, BN, false, false);  // Q, K both K-major
    constexpr uint32_t IDESC_O = ptx::idesc_f16(BF16, 2 * BM, HD, false, true);   // P K-major, V MN-major
    constexpr uint32_t DHI = ptx::sdesc_sw128_hi(1024);
    auto issue_s = [&](int x, int slot) {
      const uint32_t d = tmem + L::TM_S + x * BN;
      const uint32_t q = ptx::sdesc_sw128_lo(sQ + x * L::Q_BYTES, 16);
      const uint32_t k = ptx::sdesc_sw128_lo(sRing + slot * L::HALF_BYTES, 16);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t oq = ((kk / 4) * (BM * 128) + (kk % 4) * 32) >> 4;
        const uint32_t ok_ = ((kk / 4) * (64 * 128) + (kk % 4) * 32) >> 4;
        ptx::mma2_f16_ss(d, ptx::sdesc_join(q + oq, DHI), ptx::sdesc_join(k + ok_, DHI), IDESC_S, kk > 0 ? 1u : 0u);
      }
      ptx::mma2_commit_both(bSfull(x));
    };
    auto issue_pv = [&](int x, int slot, bool acc) {
      const uint32_t d = tmem + L::TM_O + x * HD;
      const uint32_t a = ptx::sdesc_sw128_lo(sP + x * L::P_BYTES, 16);
      const uint32_t v = ptx::sdesc_sw128_lo(sRing + slot * L::HALF_BYTES, L::HALF_BYTES);
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        const uint32_t oa = ((kk / 4) * (BM * 128) + (kk % 4) * 32) >> 4;
        ptx::mma2_f16_ss(d, ptx::sdesc_join(a + oa, DHI), ptx::sdesc_join(v + kk * ((16 * 128) >> 4), DHI), IDESC_O,
                         (acc || kk > 0) ? 1u : 0u);
      }
      ptx::mma2_commit_both(bPVdone(x));
    };
    bool ok = wait_bar_cl(bJQ, 0, abort_flag, p.watchdog_ns, WD_MMA_Q);  // both CTAs' Q and K_0
    if (ok && n > 0) {
      ptx::tc_fence_after();
      issue_s(xi, 0);
      ptx::mma2_commit_both(bEmpty(0));  // K_0
    }
    for (int j = 0; ok && j < n; ++j) {
      const int sv = (2 * j + 1) % NSLOT;  // V_j
      const int sk = (2 * j + 2) % NSLOT;  // K_{j+1}
      const bool more = j + 1 < n;
      ok = wait_bar_cl(bJPair(j % NPB), (j / NPB) & 1, abort_flag, p.watchdog_ns, WD_MMA_KV_FULL);  // V_j, K_{j+1}
      if (!ok) break;
      if (more) {  // S_X(j+1) as soon as both softmax X hold S_X(j) in registers
        ok = wait_bar_cl(bSfree(xi), j & 1, abort_flag, p.watchdog_ns, WD_MMA_S_FREE);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_s(xi, sk);
      }
      ok = wait_bar_cl(bPfull(xi), j & 1, abort_flag, p.watchdog_ns, WD_MMA_P_FULL);
      if (!ok) break;
      ptx::tc_fence_after();
      issue_pv(xi, sv, j > 0);
      ptx::mma2_commit_both(bEmpty(sv));  // V_j: this tile's P V(j) is issued (the other issuer commits too)
      if (more) ptx::mma2_commit_both(bEmpty(sk));  // K_{j+1}: this tile's S(j+1) is issued
    }
    if (ok) ptx::mma2_commit_both(bOfinal);
    // every MMA issued has finished before TMEM is freed or CTA 1's shared
    // memory goes away (the softmax may have given up without waiting for o_final)
    ptx::mma2_commit_both(bDrain);
    drain_wait(bDrain, 0, DRAIN_NS);
  }
  } else {
    ptx::setmaxnreg_inc<REGS_SOFTMAX>();
    // -------------------------------------------------------------- softmax
    const int x = warp >> 2;          // query tile of this warpgroup
    const int r = threadIdx.x & 127;  // row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + L::TM_S + x * BN;
    const uint32_t tO = tmem + lane_off + L::TM_O + x * HD;
    const uint32_t prow = sP + x * L::P_BYTES + r * 128;  // row r of P_X (and of the O staging)
    const int q0 = w.q0;
    const int hqx = w.hq[x];
    const int off = p.Skv - p.Sq;
    const int kv_all = p.causal ? min(p.Skv, off + q0 + 1) : p.Skv;       // keys every row sees
    const int row_lim = p.causal ? min(p.Skv, off + q0 + r + 1) : p.Skv;  // keys this row sees
    const float sl2 = p.sl2;
    float m_ref = -INFINITY;  // running max (log2 domain) that O and l are scaled to
    float l = 0.f;
    bool ok = true;
    auto warp_wait = [&](uint32_t b, uint32_t parity, uint32_t code) {
      return __all_sync(0xffffffffu, wait_bar_cl(b, parity, abort_flag, p.watchdog_ns, code));
    };
    for (int j = 0; j < n; ++j) {
      ok = warp_wait(bSfull(x), j & 1, WD_SOFTMAX_S_FULL);
      if (!ok) break;
      ptx::tc_fence_after();
      uint32_t sr[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) ptx::tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
      ptx::tmem_wait_ld();
      ptx::reg_fence(sr);
      // S_X is in registers: the tensor core may compute S_X(j+1) over it
      ptx::tc_fence_before();
      warp_arrive_leader<false>(bSfree(x), rank, lane);
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
      if (j > 0) {
        // P V_X(j-1) has read P_X and written O_X before this tile touches either
        ok = warp_wait(bPVdone(x), (j - 1) & 1, WD_SOFTMAX_PV_DONE);
        if (!ok) break;
        ptx::tc_fence_after();
        // the running max moved: rescale O_X in TMEM
        if (__any_sync(0xffffffffu, resc)) {
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
          ptx::tmem_wait_st();
        }
      }
      // P_X(j) into shared memory: row r, 128-byte swizzled, two 64-key blocks
      // (the layout of a K-major operand tile)
#pragma unroll
      for (int ch = 0; ch < BN / 8; ++ch)
        ptx::st_shared_v4(prow + (ch / 8) * (BM * 128) + (((ch % 8) ^ (r % 8)) * 16), pp[4 * ch], pp[4 * ch + 1],
                          pp[4 * ch + 2], pp[4 * ch + 3]);
      ptx::fence_proxy_async_smem();  // visible to the tensor core's operand reads
      ptx::tc_fence_before();
      warp_arrive_leader<true>(bPfull(x), rank, lane);
    }
    // ------------------------------------------------------------ epilogue
    // Once o_final has completed, no MMA reads P_X any more: O_X / l is staged
    // there (the layout of a Q tile) and written by TMA tensor stores, rows
    // past Sq clipped by the map.
    if (ok && n > 0) {
      ok = warp_wait(bOfinal, 0u, WD_SOFTMAX_O_DONE);
      if (ok) ptx::tc_fence_after();
    }
    if (ok) {
      if (p.lse && q0 + r < p.Sq) p.lse[(static_cast<size_t>(w.b) * p.Hq + hqx) * p.Sq + q0 + r] = row_lse(m_ref, l);
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      uint32_t orr[HD];  // the whole row: all loads in flight before one wait
      if (n > 0) {
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
        ptx::st_shared_v4(prow + (ch / 8) * (BM * 128) + (((ch % 8) ^ (r % 8)) * 16),
                          pack2<BF16>(__uint_as_float(v[0]) * inv_l, __uint_as_float(v[1]) * inv_l),
                          pack2<BF16>(__uint_as_float(v[2]) * inv_l, __uint_as_float(v[3]) * inv_l),
                          pack2<BF16>(__uint_as_float(v[4]) * inv_l, __uint_as_float(v[5]) * inv_l),
                          pack2<BF16>(__uint_as_float(v[6]) * inv_l, __uint_as_float(v[7]) * inv_l));
      }
      ptx::fence_proxy_async_smem();  // make the generic-proxy writes visible to the TMA unit
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bOstaged(x));
      if ((warp & 3) == 0) {
        ok = warp_wait(bOstaged(x), 0, WD_SOFTMAX_O_DONE);
        if (ok && lane == 0) {
          ptx::tma_store_4d(&tmO, sP + x * L::P_BYTES, 0, hqx, q0, w.b);
          ptx::tma_store_4d(&tmO, sP + x * L::P_BYTES + BM * 128, 64, hqx, q0, w.b);
          ptx::bulk_commit();
          ptx::bulk_wait_read0();  // the buffer must stay valid until the TMA unit has read it
        }
      }
    }
  }

  // ---- teardown: every role of both CTAs is done (or has drained); free TMEM
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  if (warp == MMA_WARP) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

}  // namespace fa
