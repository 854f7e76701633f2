// fa_prefill256.cuh -- the one-shot causal prefill kernel for head dimension
// 256 (sm_103a).  Included by fa_prefill.cu: it shares that file's PTX
// wrappers, bounded waits, watchdog word, Params and host helpers.
//
// At hd = 256 an O accumulator is 256 TMEM columns, so two query tiles do not
// fit in the 512 columns next to their scores.  This kernel gives a CTA ONE
// 128-row query tile and keeps P apart from S:
//
//   TMEM:  S (128 f32 columns) | P (64 columns of 16-bit pairs) | O (256 f32)
//
// With P in its own columns the MMA warp issues S(j+1) as soon as the softmax
// has read S(j) into registers, so the tensor core computes the next scores
// while the softmax works; per KV tile the tensor core has 2048 cycles of work
// (S: 128 x 128 x 256, P V: 128 x 256 x 128) against ~1100 of softmax, so one
// tile keeps it busy.
//
//   warps 0-3  softmax: one thread per row == TMEM lane (as the hd <= 128
//              kernel), S(j) -> s_free -> max / exp2 / sum -> (wait P V(j-1))
//              lazy O rescale -> P(j) -> p_full; finally O / l staged in the
//              ring and written by TMA stores
//   warp 4     tcgen05 issuer: S(0); then per KV tile j: S(j+1) after s_free(j),
//              P V(j) after p_full(j)
//   warp 5     TMA producer: Q once, then K/V in half tiles (hd columns
//              0-127 and 128-255, 32 KB each) through a ring of 5 slots, in the
//              order the MMAs consume them: K_0, then per j: K_(j+1), V_j
//   warps 6-7  idle (the CTA is two full warpgroups)

namespace fa {

constexpr int NUM_THREADS_256 = 256;
constexpr int MMA_WARP_256 = 4;
constexpr int PRODUCER_WARP_256 = 5;

struct Layout256 {
  static constexpr int HD = 256;
  static constexpr uint32_t KCH = HD / 64;                // 64-column blocks of a Q / O row
  static constexpr uint32_t Q_BYTES = BM * HD * 2;        // 64 KB
  static constexpr uint32_t HALF_BYTES = BN * 128 * 2;    // a K or V tile's 128 hd columns: 32 KB
  static constexpr int NSLOT = 5;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_RING = Q_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_RING + NSLOT * HALF_BYTES;
  // q_full, full[NSLOT], empty[NSLOT], s_full, s_free, p_full, pv_done, o_final, drain, o_staged
  static constexpr uint32_t NUM_BARS = 1 + 2 * NSLOT + 7;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;  // [0] TMEM base, [1] abort flag
  static constexpr uint32_t BYTES = OFF_MISC + 16;
  static constexpr uint32_t REQUEST = BYTES + 1024;
  static constexpr uint32_t TM_S = 0, TM_P = BN, TM_O = 256;
  static_assert(TM_P + BN / 2 <= TM_O && TM_O + HD <= TMEM_COLS, "TMEM plan");
  static_assert(OFF_RING % 1024 == 0 && HALF_BYTES % 1024 == 0, "swizzle atoms");
  static_assert(2 * HALF_BYTES == BM * HD * 2, "the O tile is staged in ring slots 0 and 1");
  static_assert(REQUEST <= 232448, "shared memory");
};

// CTA -> (batch, query head, query tile): longest tiles first; the G query
// heads of one KV group are adjacent, so their K/V tiles come from L2.
template <bool BF16>
__global__ void __launch_bounds__(NUM_THREADS_256, 1)
    fa_prefill256_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                         const Params p) {
  using L = Layout256;
  constexpr int NSLOT = L::NSLOT;
  constexpr int HD = L::HD;
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
  const uint32_t bSfull = bar + 8u * (1 + 2 * NSLOT);
  const uint32_t bSfree = bar + 8u * (2 + 2 * NSLOT);
  const uint32_t bPfull = bar + 8u * (3 + 2 * NSLOT);
  const uint32_t bPVdone = bar + 8u * (4 + 2 * NSLOT);
  const uint32_t bOfinal = bar + 8u * (5 + 2 * NSLOT);
  const uint32_t bDrain = bar + 8u * (6 + 2 * NSLOT);
  const uint32_t bOstaged = bar + 8u * (7 + 2 * NSLOT);
  uint32_t* misc = reinterpret_cast<uint32_t*>(gbase + L::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int per_qt = p.Hq * p.B;
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x / per_qt);
  const int rem = static_cast<int>(blockIdx.x % per_qt);
  const int b = rem / p.Hq;
  const int hq = rem % p.Hq;
  const int hk = hq / p.G;
  const int q0 = qt * BM;
  const int n = kv_tiles(p, q0, true);

  if (threadIdx.x == 0) {
    ptx::mbar_init(bQ, 1);
    for (int s = 0; s < NSLOT; ++s) {
      ptx::mbar_init(bFull(s), 1);
      ptx::mbar_init(bEmpty(s), 1);
    }
    ptx::mbar_init(bSfull, 1);
    ptx::mbar_init(bSfree, 4);  // one arrival per softmax warp
    ptx::mbar_init(bPfull, 4);
    ptx::mbar_init(bPVdone, 1);
    ptx::mbar_init(bOfinal, 1);
    ptx::mbar_init(bDrain, 1);
    ptx::mbar_init(bOstaged, 4);
    misc[1] = 0u;
    ptx::mbar_fence_init();
  }
  if (warp == MMA_WARP_256) {
    ptx::tmem_alloc(ptx::smem_u32(misc), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];
  // set-up overlaps the previous kernel's tail; global memory only after it
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();

  if (warp == PRODUCER_WARP_256) {
    // -------------------------------------------------------------- producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      ptx::prefetch_tmap(&tmO);
      ptx::mbar_arrive_expect_tx(bQ, L::Q_BYTES);
#pragma unroll
      for (int c = 0; c < (int)L::KCH; ++c) ptx::tma_load_4d(sQ + c * (BM * 128), &tmQ, bQ, c * 64, hq, q0, b);
      int g = 0;  // half tiles issued; half tile g goes to slot g % NSLOT
      bool ok = true;
      auto load_half = [&](const CUtensorMap* m, int t, int h) {
        const int s = g % NSLOT;
        if (g >= NSLOT) ok = wait_bar<false>(bEmpty(s), ((g / NSLOT) & 1) ^ 1u, abort_flag, p.watchdog_ns, WD_PRODUCER_EMPTY);
        if (!ok) return;
        ptx::mbar_arrive_expect_tx(bFull(s), L::HALF_BYTES);
#pragma unroll
        for (int c = 0; c < 2; ++c)
          ptx::tma_load_4d(sRing + s * L::HALF_BYTES + c * (BN * 128), m, bFull(s), (2 * h + c) * 64, hk, t * BN, b);
        ++g;
      };
      if (n > 0) {
        load_half(&tmK, 0, 0);
        if (ok) load_half(&tmK, 0, 1);
      }
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) {
          load_half(&tmK, j + 1, 0);
          if (ok) load_half(&tmK, j + 1, 1);
        }
        if (ok) load_half(&tmV, j, 0);
        if (ok) load_half(&tmV, j, 1);
      }
      // every copy issued has landed before the CTA exits (as in the two-tile kernel)
      drain_wait(bQ, 0, DRAIN_NS);
      for (int s = 0; s < NSLOT && s < g; ++s) {
        const int last = s + NSLOT * ((g - 1 - s) / NSLOT);
        drain_wait(bFull(s), (last / NSLOT) & 1, DRAIN_NS);
      }
    }
  } else if (warp == MMA_WARP_256) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = ptx::idesc_f16(BF16, BM, BN, false, false);   // Q, K both K-major
      constexpr uint32_t IDESC_O = ptx::idesc_f16(BF16, BM, 128, false, true);   // P from TMEM, V MN-major
      constexpr uint32_t DHI = ptx::sdesc_sw128_hi(1024);  // Q, K (K-major) and V (MN-major): SBO 1024
      int g = 0;  // half tiles consumed, in load order
      bool ok = true;
      auto half_ready = [&]() -> int {
        const int s = g % NSLOT;
        ok = wait_bar<false>(bFull(s), (g / NSLOT) & 1, abort_flag, p.watchdog_ns, WD_MMA_KV_FULL);
        return s;
      };
      auto issue_s = [&]() {  // S = Q K^T over both hd halves, slot by slot
        for (int h = 0; ok && h < 2; ++h) {
          const int s = half_ready();
          if (!ok) return;
          ptx::tc_fence_after();
          const uint32_t q = ptx::sdesc_sw128_lo(sQ, 16);
          const uint32_t k = ptx::sdesc_sw128_lo(sRing + s * L::HALF_BYTES, 16);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // 16 hd columns per MMA
            const uint32_t oq = ((2 * h + kk / 4) * (BM * 128) + (kk % 4) * 32) >> 4;
            const uint32_t ok_ = ((kk / 4) * (BN * 128) + (kk % 4) * 32) >> 4;
            ptx::mma_f16_ss(tmem + L::TM_S, ptx::sdesc_join(q + oq, DHI), ptx::sdesc_join(k + ok_, DHI), IDESC_S,
                            (h > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(bEmpty(s));
          ++g;
        }
        if (ok) ptx::mma_commit(bSfull);
      };
      auto issue_pv = [&](bool acc) {  // O[:, 128 h ...] += P V[:, 128 h ...], slot by slot
        for (int h = 0; ok && h < 2; ++h) {
          const int s = half_ready();
          if (!ok) return;
          ptx::tc_fence_after();
          const uint32_t v = ptx::sdesc_sw128_lo(sRing + s * L::HALF_BYTES, BN * 128);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            ptx::mma_f16_ts(tmem + L::TM_O + h * 128, tmem + L::TM_P + kk * 8,
                            ptx::sdesc_join(v + kk * ((16 * 128) >> 4), DHI), IDESC_O, (acc || kk > 0) ? 1u : 0u);
          ptx::mma_commit(bEmpty(s));
          ++g;
        }
        if (ok) ptx::mma_commit(bPVdone);
      };
      ok = wait_bar<false>(bQ, 0, abort_flag, p.watchdog_ns, WD_MMA_Q);
      if (ok && n > 0) issue_s();
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) {  // S(j+1) once the softmax holds S(j) in registers
          ok = wait_bar<false>(bSfree, j & 1, abort_flag, p.watchdog_ns, WD_MMA_P_FULL);
          if (!ok) break;
          issue_s();
          if (!ok) break;
        }
        ok = wait_bar<false>(bPfull, j & 1, abort_flag, p.watchdog_ns, WD_MMA_P_FULL);
        if (!ok) break;
        issue_pv(j > 0);
      }
      if (ok) ptx::mma_commit(bOfinal);
      ptx::mma_commit(bDrain);  // every MMA issued has finished before TMEM is freed
      drain_wait(bDrain, 0, DRAIN_NS);
    }
  } else if (warp < 4) {
    // -------------------------------------------------------------- softmax
    const int r = threadIdx.x;  // row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off + L::TM_S;
    const uint32_t tP = tmem + lane_off + L::TM_P;
    const uint32_t tO = tmem + lane_off + L::TM_O;
    const int off = p.Skv - p.Sq;
    const int kv_all = p.causal ? min(p.Skv, off + q0 + 1) : p.Skv;
    const int row_lim = p.causal ? min(p.Skv, off + q0 + r + 1) : p.Skv;
    const float sl2 = p.sl2;
    float m_ref = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      ok = warp_wait_bar<false>(bSfull, j & 1, abort_flag, p.watchdog_ns, WD_SOFTMAX_S_FULL);
      if (!ok) break;
      ptx::tc_fence_after();
      uint32_t sr[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) ptx::tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
      ptx::tmem_wait_ld();
      ptx::reg_fence(sr);
      ptx::tc_fence_before();  // S(j) is in registers: S(j+1) may overwrite it
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bSfree);
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
      const float mx = ptx::fmax3(ptx::fmax3(mk[0], mk[1], mk[2]), ptx::fmax3(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7]));
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
      if (j > 0) {  // P(j-1) consumed and O updated before P(j) and a rescale
        ok = warp_wait_bar<false>(bPVdone, (j - 1) & 1, abort_flag, p.watchdog_ns, WD_SOFTMAX_O_DONE);
        if (!ok) break;
        ptx::tc_fence_after();
        if (__any_sync(0xffffffffu, resc)) {
          const uint64_t a2 = ptx::pk(alpha, alpha);
#pragma unroll 1
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
      ptx::tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&pp[0]));
      ptx::tmem_st32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&pp[32]));
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bPfull);
    }
    // ------------------------------------------------------------ epilogue
    // After o_final every half tile loaded was consumed: ring slots 0 and 1
    // (64 KB, contiguous) stage O, written out by one TMA store per 64 columns.
    if (ok && n > 0) {
      ok = warp_wait_bar<false>(bOfinal, 0, abort_flag, p.watchdog_ns, WD_SOFTMAX_O_DONE);
      if (ok) ptx::tc_fence_after();
    }
    if (ok) {
      if (p.lse && q0 + r < p.Sq) p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.Sq + q0 + r] = row_lse(m_ref, l);
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const uint32_t stage = sRing + r * 128;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t orr[32];
        if (n > 0) {
          ptx::tmem_ld32(tO + c * 32, orr);
          ptx::tmem_wait_ld();
          ptx::reg_fence(orr);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = 0u;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int ch = c * 4 + e;  // 16-byte chunk of the row
          ptx::st_shared_v4(stage + (ch / 8) * (BM * 128) + (((ch % 8) ^ (r % 8)) * 16),
                            pack2<BF16>(__uint_as_float(orr[8 * e + 0]) * inv_l, __uint_as_float(orr[8 * e + 1]) * inv_l),
                            pack2<BF16>(__uint_as_float(orr[8 * e + 2]) * inv_l, __uint_as_float(orr[8 * e + 3]) * inv_l),
                            pack2<BF16>(__uint_as_float(orr[8 * e + 4]) * inv_l, __uint_as_float(orr[8 * e + 5]) * inv_l),
                            pack2<BF16>(__uint_as_float(orr[8 * e + 6]) * inv_l, __uint_as_float(orr[8 * e + 7]) * inv_l));
        }
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bOstaged);
      if (warp == 0) {
        ok = warp_wait_bar<false>(bOstaged, 0, abort_flag, p.watchdog_ns, WD_SOFTMAX_O_DONE);
        if (ok && lane == 0) {
#pragma unroll
          for (int c = 0; c < (int)L::KCH; ++c)  // a narrower head has no columns past p.hd: no store there
            if (c * 64 < p.hd) ptx::tma_store_4d(&tmO, sRing + c * (BM * 128), c * 64, hq, q0, b);
          ptx::bulk_commit();
          ptx::bulk_wait_read0();
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP_256) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace fa
