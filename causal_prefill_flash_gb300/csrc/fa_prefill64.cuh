// fa_prefill64.cuh -- the one-shot kernel for heads up to 64 wide, with S and
// P in separate TMEM columns (included by fa_prefill.cu).
//
// The per-tile steps are the pages' (minfer "53 · r50 — FA_TKV 32->16
// occupancy experiment", section 2: S = Q K^T, mask, max, exp, sum, rescale O,
// O += P V), planned as in the 128-wide kernel: one CTA owns two 128-row
// query tiles A and B that read the same K/V, a TMA producer, one MMA warp,
// a softmax warpgroup per tile (one thread per row == TMEM lane).
//
// What differs: at hd 64 the two S tiles (2 x 128 columns) and the two O
// accumulators (2 x 64) leave 128 TMEM columns free, exactly the two P tiles
// (128 x 128 16-bit = 64 columns each).  So P does not overwrite S, and the
// MMA warp issues S_X(j+1) as soon as softmax X has read S_X(j) into its
// registers (an s_free barrier), not after P V_X(j): the next tile's S is
// computed while the softmax still works on this one, and the MMA and its
// hand-offs drop out of the tile's chain.  In exchange, softmax X waits for
// P V_X(j-1) to complete (a pv_done barrier) before it rescales O_X or
// writes P_X(j) -- which by then it has, a whole softmax later.
//
//   TMEM (512 columns): S_A | S_B | O_A | O_B | P_A | P_B
//                       128   128   64    64    64    64
//
// Per KV step j the MMA warp issues, for X = A, B:
//   S_X(j+1) once s_free_X(j), then P V_X(j) once p_full_X(j).
// The K/V ring, its pair barriers and per-slot frees, the staged TMA-store
// epilogue, programmatic dependent launch and the bounded waits are those of
// the 128-wide kernel.  The MMA warp runs its loop converged, one elected
// lane issuing (its N = 64 P V MMAs make the issue rate matter).

namespace fa {

// Watchdog codes of this kernel (bits 0-7 of g_fa_status), beside the shared ones.
enum : uint32_t {
  WD_MMA_S_FREE = 10,       // the MMA warp waiting for a softmax to have read S
  WD_SOFTMAX_PV_DONE = 11,  // a softmax waiting for the previous P V of its tile
};

struct Layout64 {
  using L = Layout<64>;
  static constexpr uint32_t KCH = 1;                 // one 128-byte column block along hd
  static constexpr uint32_t Q_BYTES = L::Q_BYTES;    // 16 KB
  static constexpr uint32_t SLOT_BYTES = L::SLOT_BYTES;
  static constexpr int NSLOT = 8;                    // K/V ring depth
  static constexpr int NPB = (NSLOT + 1) / 2;        // (V_j, K_j+1) pair barriers
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_RING = 2 * Q_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_RING + NSLOT * SLOT_BYTES;
  // q_full (Q and K_0), pair[NPB], empty[NSLOT], s_full[2], s_free[2], p_full[2],
  // pv_done[2], o_final, drain, o_staged[2]
  static constexpr uint32_t NUM_BARS = 1 + NPB + NSLOT + 2 + 2 + 2 + 2 + 1 + 1 + 2;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;  // [0] TMEM base, [1] abort flag
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static constexpr uint32_t REQUEST = BYTES + 1024;  // slack to align the dynamic base
  static constexpr uint32_t TM_S = 0;        // S_A, S_B: 128 columns each
  static constexpr uint32_t TM_O = 2 * BN;   // O_A, O_B: 64 columns each
  static constexpr uint32_t TM_P = TM_O + 2 * 64;  // P_A, P_B: 64 columns each
  static_assert(TM_P + 2 * (BN / 2) <= TMEM_COLS, "TMEM plan");
  static_assert(OFF_RING % 1024 == 0 && SLOT_BYTES % 1024 == 0, "swizzle atoms");
  static_assert(2 * NPB >= NSLOT, "pair barriers");
};

template <bool BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fa_prefill64_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                        const __grid_constant__ CUtensorMap tmKt, const __grid_constant__ CUtensorMap tmVt,
                        const Params p) {
  constexpr int HD = 64;
  using L = Layout64;
  constexpr int NSLOT = L::NSLOT;
  constexpr int NPB = L::NPB;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);

  const uint32_t sQ = sbase + L::OFF_Q;
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
      ptx::mbar_init(bSfree(x), BM);  // every softmax thread of the tile, once its S row is in registers
      ptx::mbar_init(bPfull(x), BM);  // every softmax thread of the tile, once its P row is in TMEM
      ptx::mbar_init(bPVdone(x), 1);
    }
    ptx::mbar_init(bOfinal, 1);
    ptx::mbar_init(bDrain, 1);
    ptx::mbar_init(bOstaged(0), 4);  // one arrival per softmax warp of the tile
    ptx::mbar_init(bOstaged(1), 4);
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
  // the set-up above overlaps the previous kernel's tail; nothing in global
  // memory is read or written before that kernel has completed
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();

  if (warp >= MMA_WARP) {
  ptx::setmaxnreg_dec<REGS_CONTROL>();
  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    // as in the 128-wide kernel: Q_A, Q_B and K_0 on the Q barrier, then
    // V_j and K_j+1 on pair barrier j % NPB; load i in slot i % NSLOT, each
    // slot freed by its own commit
    if (lane == 0) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      ptx::prefetch_tmap(&tmO);
      ptx::mbar_arrive_expect_tx(bQ, L::Q_BYTES * (w.has[1] ? 2u : 1u) + (n > 0 ? L::SLOT_BYTES : 0u));
      for (int x = 0; x < 2; ++x) {
        if (!w.has[x]) continue;
        ptx::tma_load_4d(sQ + x * L::Q_BYTES, &tmQ, bQ, 0, w.hq[x], w.q0[x], w.b);
      }
      int issued = 0;
      bool ok = true;
      int page = -1, blk = 0;  // paged K/V: the pool block of the current page
      if (p.block_table) {
        ptx::prefetch_tmap(&tmKt);
        ptx::prefetch_tmap(&tmVt);
      }
      for (int i = 0; i < 2 * n; ++i) {
        const int s = i % NSLOT;
        if (i >= NSLOT) ok = wait_bar(bEmpty(s), ((i / NSLOT) & 1) ^ 1u, abort_flag, p.watchdog_ns, WD_PRODUCER_EMPTY);
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
        ptx::tma_load_4d(sRing + s * L::SLOT_BYTES, m, fb, 0, w.hk, row, bat);
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
  } else if (warp == MMA_WARP) {
    // ----------------------------------------------------------- MMA issuer
    // the whole warp runs the loop and the waits; one elected lane issues
    const bool leader = ptx::elect_one();
    constexpr uint32_t IDESC_S = ptx::idesc_f16(BF16, BM, BN, false, false);  // Q, K both K-major
    constexpr uint32_t IDESC_O = ptx::idesc_f16(BF16, BM, HD, false, true);   // P from TMEM, V MN-major
    constexpr uint32_t DHI = ptx::sdesc_sw128_hi(1024);
    auto issue_s = [&](int x, int slot) {
      const uint32_t d = tmem + L::TM_S + x * BN;
      const uint32_t q = ptx::sdesc_sw128_lo(sQ + x * L::Q_BYTES, 16);
      const uint32_t k = ptx::sdesc_sw128_lo(sRing + slot * L::SLOT_BYTES, 16);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t o = ((kk % 4) * 32) >> 4;
        if (leader) ptx::mma_f16_ss(d, ptx::sdesc_join(q + o, DHI), ptx::sdesc_join(k + o, DHI), IDESC_S, kk > 0 ? 1u : 0u);
      }
      if (leader) ptx::mma_commit(bSfull(x));
    };
    auto issue_pv = [&](int x, int slot, bool acc) {
      const uint32_t d = tmem + L::TM_O + x * HD;
      const uint32_t a = tmem + L::TM_P + x * (BN / 2);  // P_X, 2 elements per column
      const uint32_t v = ptx::sdesc_sw128_lo(sRing + slot * L::SLOT_BYTES, BN * 128);
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk)
        if (leader)
          ptx::mma_f16_ts(d, a + kk * 8, ptx::sdesc_join(v + kk * ((16 * 128) >> 4), DHI), IDESC_O,
                          (acc || kk > 0) ? 1u : 0u);
      if (leader) ptx::mma_commit(bPVdone(x));
    };
    bool ok = warp_wait_bar(bQ, 0, abort_flag, p.watchdog_ns, WD_MMA_Q);  // Q and K_0
    if (ok && n > 0) {
      ptx::tc_fence_after();
      if (nA > 0) issue_s(0, 0);
      if (nB > 0) issue_s(1, 0);
      if (leader) ptx::mma_commit(bEmpty(0));  // K_0
    }
    for (int j = 0; ok && j < n; ++j) {
      const int iv = 2 * j + 1, sv = iv % NSLOT;  // V_j
      const int ik = 2 * j + 2, sk = ik % NSLOT;  // K_{j+1}
      const bool more = j + 1 < n;
      ok = warp_wait_bar(bPair(j % NPB), (j / NPB) & 1, abort_flag, p.watchdog_ns, WD_MMA_KV_FULL);  // V_j, K_{j+1}
      if (!ok) break;
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int nX = x == 0 ? nA : nB;
        if (j < nX) {
          if (j + 1 < nX) {  // S_X(j+1) as soon as softmax X holds S_X(j) in registers
            ok = warp_wait_bar(bSfree(x), j & 1, abort_flag, p.watchdog_ns, WD_MMA_S_FREE);
            if (!ok) break;
            ptx::tc_fence_after();
            issue_s(x, sk);
          }
          ok = warp_wait_bar(bPfull(x), j & 1, abort_flag, p.watchdog_ns, WD_MMA_P_FULL);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_pv(x, sv, j > 0);
        }
      }
      if (!ok) break;
      if (leader) ptx::mma_commit(bEmpty(sv));  // V_j: both tiles' P V(j) are issued
      if (more && leader) ptx::mma_commit(bEmpty(sk));  // K_{j+1}: both tiles' S(j+1) are issued
    }
    if (ok && leader) ptx::mma_commit(bOfinal);
    // every MMA issued has finished before TMEM is freed (the softmax may
    // have given up without waiting for o_final)
    if (leader) ptx::mma_commit(bDrain);
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
    const uint32_t tP = tmem + lane_off + L::TM_P + x * (BN / 2);
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
      // S_X is in registers: the tensor core may compute S_X(j+1) over it
      ptx::tc_fence_before();
      ptx::mbar_arrive(bSfree(x));
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
        ok = warp_wait_bar(bPVdone(x), (j - 1) & 1, abort_flag, p.watchdog_ns, WD_SOFTMAX_PV_DONE);
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
        }
      }
      // P_X(j) into its own columns
      ptx::tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&pp[0]));
      ptx::tmem_st32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&pp[32]));
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bPfull(x));
    }
    // ------------------------------------------------------------ epilogue
    // Once o_final has completed, no MMA reads the ring any more (waited
    // whenever the CTA streams any KV tile, even if this tile has none).
    if (ok && n > 0) {
      ok = warp_wait_bar(bOfinal, 0u, abort_flag, p.watchdog_ns, WD_SOFTMAX_O_DONE);
      if (ok) ptx::tc_fence_after();
    }
    if (ok && hasx) {
      if (p.lse && q0 + r < p.Sq) p.lse[(static_cast<size_t>(w.b) * p.Hq + hqx) * p.Sq + q0 + r] = row_lse(m_ref, l);
      // O / l rounded to 16 bits, written 128-byte swizzled into a ring slot no
      // MMA reads any more and sent out by a TMA tensor store (rows past Sq
      // clipped by the map)
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const int stage_slot = (2 * n + 2 * NSLOT - 4 + x) % NSLOT;
      const uint32_t stage = sRing + stage_slot * L::SLOT_BYTES + r * 128;
      uint32_t orr[HD];
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
        ptx::st_shared_v4(stage + (((ch % 8) ^ (r % 8)) * 16),
                          pack2<BF16>(__uint_as_float(v[0]) * inv_l, __uint_as_float(v[1]) * inv_l),
                          pack2<BF16>(__uint_as_float(v[2]) * inv_l, __uint_as_float(v[3]) * inv_l),
                          pack2<BF16>(__uint_as_float(v[4]) * inv_l, __uint_as_float(v[5]) * inv_l),
                          pack2<BF16>(__uint_as_float(v[6]) * inv_l, __uint_as_float(v[7]) * inv_l));
      }
      ptx::fence_proxy_async_smem();  // make the generic-proxy writes visible to the TMA unit
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bOstaged(x));
      if ((warp & 3) == 0) {
        ok = warp_wait_bar(bOstaged(x), 0, abort_flag, p.watchdog_ns, WD_SOFTMAX_O_DONE);
        if (ok && lane == 0) {
          ptx::tma_store_4d(&tmO, sRing + stage_slot * L::SLOT_BYTES, 0, hqx, q0, w.b);
          ptx::bulk_commit();
          ptx::bulk_wait_read0();  // the slot must stay valid until the TMA unit has read it
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

}  // namespace fa
