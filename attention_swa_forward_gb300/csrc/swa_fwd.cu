// swa_fwd.cu — sliding-window attention forward on sm_103a.
//
// Computes, per query row i (FlashAttentionVarLenScore doc, "计算公式"):
//   O_i = sum_j softmax_j(scale * q_i.k_j over visible j) * z_ij / keep * v_j
// plus softmax_max_i and softmax_sum_i (before dropout), with the online
// (blockwise) softmax of the PyPTO-Gym article's forward ("前向公式"; the
// statistics it saves for the backward).
//
// One CTA = one 128-row query tile of one (batch, head); it walks only the
// 128-key tiles that intersect the BAND window.  Warp roles:
//   warps 0-3  softmax + epilogue, one thread per query row (TMEM lane)
//   warp  4    TMA producer: Q once; K and V through separate 3-stage rings
//              (a K stage is released as soon as its S is computed)
//   warp  5    tcgen05 issuer of S = Q K^T into a double-buffered TMEM tile
//   warp  6    tcgen05 issuer of O += P V, P (bf16) taken from TMEM as the
//              A operand
// Two issuing threads keep the tensor pipe fed: its queue is shallow, so
// every barrier wait of a single issuer between GEMMs left it idle; with two,
// one waits while the other's GEMM runs.
// TMEM columns: S0 [0,128), S1 [128,256), O [256,256+D), P0 [384,448),
// P1 [448,512).
#include "swa_device.cuh"

namespace swa {
namespace {

constexpr int kStages = 3;

template <int D>
struct FwdSmem {
  static constexpr int kTileBytes = kTileM * D * 2;
  alignas(1024) uint8_t q[kTileBytes];
  alignas(1024) uint8_t k[kStages][kTileBytes];
  alignas(1024) uint8_t v[kStages][kTileBytes];
  uint64_t q_full, k_full[kStages], v_full[kStages], k_empty[kStages], v_empty[kStages];
  uint64_t s_full[2], s_free[2], p_full[2], o_done[2], drain_s, drain_pv;  // o_done[b]: PV of P buffer b
  uint64_t never;  // completed by nothing: the target of the stall test hook
  uint32_t tmem_base;
};
static_assert(sizeof(FwdSmem<128>) + 1024 <= 232448, "shared memory budget");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256, kColP = 384;  // P buffer b at kColP + 64*b
constexpr float kLn2 = 0.6931471805599453f;
// Rescale O only when the running max grows by more than 2^8 (log2 units);
// until then the stale max is kept and p may reach 256, far from overflow.
constexpr float kRescaleThreshold = 8.0f;

template <int D, int DM, bool F16, int CAP>
__global__ void __launch_bounds__(224, 1)
    swa_fwd_kernel(const FwdArgs a, const __grid_constant__ SeqTable<CAP> tab, const __grid_constant__ CUtensorMap mq,
                   const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv) {
  extern __shared__ uint8_t smem_raw[];
  FwdSmem<D>& s = *reinterpret_cast<FwdSmem<D>*>(align1024(smem_raw));
  constexpr int kTileBytes = FwdSmem<D>::kTileBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // q, k, v, the outputs and the status word may belong to the previous grid
  // on the stream (this kernel is launched with programmatic serialization):
  // wait for it before touching any of them.  No early trigger: the next
  // grid starts when this one ends (backward CTAs made resident during the
  // forward's last wave slowed the whole step)
  griddep_wait();
  if (a.clear_err && blockIdx.x == 0 && threadIdx.x == 0) *a.err = 0;
  const Geometry& g = a.g;
  const Item w = resolve_item(tab, a.g, static_cast<int>(blockIdx.x), a.g.N);
  const int hk = w.n / a.g.group;  // the key/value head this query head reads
  const SeqInfo sq = w.s;
  const int q0 = w.tile * kTileM;

  // key tiles touched by this query tile
  int kv_t0, n_kv;
  key_tiles_of_query_tile(g, sq, w.tile, &kv_t0, &n_kv);

  // The producer's lane initialises the barriers and issues the loads of Q
  // and the first K tile before the CTA-wide barrier, so their latency runs
  // while TMEM is allocated.
  if (warp == 4 && lane == 0) {
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
      mbar_init(&s.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_free[i], kTileM);
      mbar_init(&s.p_full[i], kTileM);
    }
    mbar_init(&s.o_done[0], 1);
    mbar_init(&s.o_done[1], 1);
    mbar_init(&s.drain_s, 1);
    mbar_init(&s.drain_pv, 1);
    mbar_init(&s.never, 1);
    fence_mbar_init();
    if (n_kv > 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
      mbar_arrive_expect_tx(&s.q_full, kTileBytes);
      tma_rows<D>(s.q, &mq, &s.q_full, g, w.b, w.n, sq.q_start, q0);
      mbar_arrive_expect_tx(&s.k_full[0], kTileBytes);
      tma_rows<D>(s.k[0], &mk, &s.k_full[0], g, w.b, hk, sq.kv_start, kv_t0 * kTileN);
    }
  }
  if (warp == 5) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s.tmem_base;

  if (warp == 4) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0 && n_kv > 0) {
      int k_issued = 1, v_issued = 0;  // Q and K(0) went out before the CTA-wide barrier
      for (int it = 0; it < n_kv; ++it) {
        const int st = it % kStages;
        const uint32_t use = it / kStages;
        const int j0 = (kv_t0 + it) * kTileN;
        if (it > 0) {
          if (it >= kStages && !mbar_wait(&s.k_empty[st], (use - 1) & 1, a.err, kErrFwdLoad)) break;
          mbar_arrive_expect_tx(&s.k_full[st], kTileBytes);
          tma_rows<D>(s.k[st], &mk, &s.k_full[st], g, w.b, hk, sq.kv_start, j0);
          ++k_issued;
        }
        if (it >= kStages && !mbar_wait(&s.v_empty[st], (use - 1) & 1, a.err, kErrFwdLoad)) break;
        mbar_arrive_expect_tx(&s.v_full[st], kTileBytes);
        tma_rows<D>(s.v[st], &mv, &s.v_full[st], g, w.b, hk, sq.kv_start, j0);
        ++v_issued;
      }
      // every copy issued has landed before the CTA may exit
      mbar_wait_drain(&s.q_full, 0);
      for (int st = 0; st < kStages; ++st) {
        const int uk = (k_issued - st + kStages - 1) / kStages, uv = (v_issued - st + kStages - 1) / kStages;
        if (uk > 0) mbar_wait_drain(&s.k_full[st], (uk - 1) & 1);
        if (uv > 0) mbar_wait_drain(&s.v_full[st], (uv - 1) & 1);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------ S = Q K^T issuer --
    if (lane == 0 && n_kv > 0) {
      constexpr uint32_t kIdS = idesc_f16_f32(kTileM, kTileN, false, false, F16);
      const uint32_t q_addr = smem_u32(s.q);
      const int nk = d_steps(g);
      bool ok = mbar_wait(&s.q_full, 0, a.err, kErrFwdMma);
      for (int it = 0; ok && it < n_kv; ++it) {
        const int st = it % kStages, sb = it & 1;
        // S buffer sb was last read by the softmax of tile it - 2
        if (it >= 2 && !mbar_wait(&s.s_free[sb], ((it >> 1) - 1) & 1, a.err, kErrFwdMma)) break;
        if (!mbar_wait(&s.k_full[st], (it / kStages) & 1, a.err, kErrFwdMma)) break;
        tc_fence_after_sync();
        const uint64_t dq_ = sdesc_sw128(q_addr, 16, 1024), dk_ = sdesc_sw128(smem_u32(s.k[st]), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          if (kk >= nk) break;
          const uint32_t off = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
          umma_bf16_ss(tmem + sb * kTileN, sdesc_advance(dq_, off), sdesc_advance(dk_, off), kIdS, kk > 0);
        }
        umma_commit(&s.s_full[sb]);
        umma_commit(&s.k_empty[st]);
      }
      umma_commit(&s.drain_s);
      mbar_wait_drain(&s.drain_s, 0);
    }
  } else if (warp == 6) {
    // ------------------------------------------------- O += P V issuer --
    if (lane == 0 && n_kv > 0) {
      constexpr uint32_t kIdO = idesc_f16_f32(kTileM, D, false, true, F16);
      for (int it = 0; it < n_kv; ++it) {
        const int pb = it & 1, st = it % kStages;
        if (!mbar_wait(&s.p_full[pb], (it >> 1) & 1, a.err, kErrFwdMma)) break;
        if (!mbar_wait(&s.v_full[st], (it / kStages) & 1, a.err, kErrFwdMma)) break;
        tc_fence_after_sync();
        const uint64_t dv_ = sdesc_sw128(smem_u32(s.v[st]), kAtomBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk)  // O += P V  (A = P in TMEM)
          umma_bf16_ts(tmem + kColO, tmem + kColP + pb * 64 + kk * 8, sdesc_advance(dv_, kk * 2048), kIdO,
                       (it > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&s.o_done[pb]);
        umma_commit(&s.v_empty[st]);
      }
      umma_commit(&s.drain_pv);
      mbar_wait_drain(&s.drain_pv, 0);
    }
  } else {
    // ------------------------------------------ softmax + epilogue (rows) --
    const int r = threadIdx.x;  // 0..127 == TMEM lane
    const int i = q0 + r;
    const bool row_valid = i < sq.q_len;
    int wlo, whi;
    key_window(g, sq, i, wlo, whi);
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float c = g.scale_log2;
    float m_use = -INFINITY, m_true = -INFINITY, l = 0.f;
    bool ok = true;
    // test hook: wait on a barrier that nothing completes, so the bounded
    // wait runs out and the launch reports it
    if (g.stall & kStallForward)
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(&s.never, 0, a.err, kErrFwdSoftmax));
    bool s_ready = false;  // S(it) known complete from a probe issued during the previous tile
    // Keep bits read from the mask are fetched one tile ahead, so their
    // global-load latency is not on the softmax's path.
    uint32_t next_bits[4] = {0u, 0u, 0u, 0u};
    if (DM == 1 && n_kv > 0 && row_valid) load_keep_bits(a.mask, sq, w.n, i, kv_t0 * kTileN, next_bits, g.n_mask_bytes, a.err);
    for (int it = 0; ok && it < n_kv; ++it) {
      const int sb = it & 1;
      uint32_t bits[4] = {~0u, ~0u, ~0u, ~0u};
      if (DM == 1) {
#pragma unroll
        for (int u = 0; u < 4; ++u) bits[u] = next_bits[u];
        if (it + 1 < n_kv && row_valid) load_keep_bits(a.mask, sq, w.n, i, (kv_t0 + it + 1) * kTileN, next_bits, g.n_mask_bytes, a.err);
      }
      // warp-uniform outcome: the tcgen05.ld below is warp-collective
      if (!s_ready && !__all_sync(0xFFFFFFFFu, mbar_wait(&s.s_full[sb], (it >> 1) & 1, a.err, kErrFwdSoftmax))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      // the row's 128 scores, loaded in place (xr holds fp32 bits, later the bf16 P pairs)
      uint32_t xr[kTileN];
      {
        uint32_t(&x0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&xr[0]);
        uint32_t(&x1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&xr[32]);
        uint32_t(&x2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&xr[64]);
        uint32_t(&x3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&xr[96]);
        const uint32_t base = tmem + lane_off + sb * kTileN;
        tmem_ld_32x32b_x32(base + 0, x0);  // all four loads in flight before the one wait
        tmem_ld_32x32b_x32(base + 32, x1);
        tmem_ld_32x32b_x32(base + 64, x2);
        tmem_ld_32x32b_x32(base + 96, x3);
        tmem_ld_wait(x0);
        tmem_ld_wait(x1);
        tmem_ld_wait(x2);
        tmem_ld_wait(x3);
      }
      tc_fence_before_sync();
      mbar_arrive(&s.s_free[sb]);
      // P buffer sb was last read by PV(it-2): probe now, use the answer
      // after the exponentials
      const bool p_free = it < 2 || mbar_test(&s.o_done[sb], ((it >> 1) - 1) & 1);
      auto X = [&](int t) -> float { return __uint_as_float(xr[t]); };

      const int j0 = (kv_t0 + it) * kTileN;
      // With a positive scale the maximum is taken on the raw scores and the
      // scale folds into one packed FMA per pair, p = exp2(x*c - m); keys
      // outside the window (partial tiles only) become -inf first, and
      // exp2(-inf*c - m) = 0.  A scale <= 0 takes scale, mask, exp2(x - m).
      const bool fold = c > 0.f;
      const bool fast = fold && tile_fully_visible(g, sq, q0, j0);
      float mx;
      {
        float m8[8];  // eight independent partial maxima: no long dependency chain
#pragma unroll
        for (int u = 0; u < 8; ++u) m8[u] = -INFINITY;
        if (fast) {
#pragma unroll
          for (int t = 0; t < kTileN; t += 2) m8[(t >> 1) & 7] = fmax3(m8[(t >> 1) & 7], X(t), X(t + 1));
        } else {
          const int lo_t = wlo - j0, hi_t = whi - j0;  // visible t in [lo_t, hi_t]
#pragma unroll
          for (int t = 0; t < kTileN; ++t) {
            const bool vis = (t >= lo_t) & (t <= hi_t);
            const float v = vis ? (fold ? X(t) : X(t) * c) : -INFINITY;  // selects, not branches
            xr[t] = __float_as_uint(v);
            m8[t & 7] = fmaxf(m8[t & 7], v);
          }
        }
        mx = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], fmax3(m8[5], m8[6], m8[7])));
        if (fold) mx *= c;
      }
      const float m_new = fmaxf(m_true, mx);
      m_true = m_new;
      const bool need = m_new > m_use + kRescaleThreshold;
      const bool warp_need = __any_sync(0xFFFFFFFFu, need);
      float alpha = 1.f;
      if (need) {
        alpha = ex2_approx(m_use - m_new);
        m_use = m_new;
      }
      const float msub = (m_use == -INFINITY) ? 0.f : m_use;
      if (DM == 2) gen_keep_words<4>(g, stat_index(g, sq, w.b, w.n, i), j0 >> 4, bits);
      // p = exp2(.), the row sum of p (before dropout), then P = p*z packed
      // to bf16 pairs in place: xr[t/2] receives the pair (t, t+1)
      float r8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) r8[u] = 0.f;
#pragma unroll
      for (int t = 0; t < kTileN; t += 2) {
        float p0, p1;
        if (fold) {
          ffma2_bcast(p0, p1, X(t), X(t + 1), c, -msub);
        } else {
          p0 = X(t) - msub;
          p1 = X(t + 1) - msub;
        }
        p0 = ex2_approx(p0);
        p1 = ex2_approx(p1);
        fadd2_acc(r8[(t >> 1) & 3], r8[4 + ((t >> 1) & 3)], p0, p1);
        if (DM != 0) {
          p0 = ((bits[t >> 5] >> (t & 31)) & 1u) ? p0 : 0.f;
          p1 = ((bits[(t + 1) >> 5] >> ((t + 1) & 31)) & 1u) ? p1 : 0.f;
        }
        xr[t >> 1] = pack2<F16>(p0, p1);
      }
      const float rs = ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
      l = l * alpha + rs;
      // P buffer (it & 1) was last read by PV(it-2).  Only a warp that must
      // rescale its rows of O also waits for PV(it-1); the others write P(it)
      // while PV(it-1) may still run, so the tensor pipe never waits for the
      // softmax's hand-off in the common case.
      if (!__all_sync(0xFFFFFFFFu, p_free) &&
          !__all_sync(0xFFFFFFFFu, mbar_wait(&s.o_done[sb], ((it >> 1) - 1) & 1, a.err, kErrFwdSoftmax))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      if (it >= 1 && warp_need) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&s.o_done[sb ^ 1], ((it - 1) >> 1) & 1, a.err, kErrFwdSoftmax))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        {
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t t32[32];
            const uint32_t addr = tmem + lane_off + kColO + ch * 32;
            tmem_ld_32x32b_x32(addr, t32);
            tmem_ld_wait(t32);
#pragma unroll
            for (int t = 0; t < 32; ++t) t32[t] = __float_as_uint(__uint_as_float(t32[t]) * alpha);
            tmem_st_32x32b_x32(addr, t32);
          }
        }
      }
      // probe the next tile's S while P is stored; the answer is used at the top of the next tile
      const bool s_next = it + 1 < n_kv && mbar_test(&s.s_full[sb ^ 1], ((it + 1) >> 1) & 1);
      tmem_st_32x32b_x32(tmem + lane_off + kColP + sb * 64, *reinterpret_cast<const uint32_t(*)[32]>(&xr[0]));
      tmem_st_32x32b_x32(tmem + lane_off + kColP + sb * 64 + 32, *reinterpret_cast<const uint32_t(*)[32]>(&xr[32]));
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&s.p_full[sb]);
      s_ready = __all_sync(0xFFFFFFFFu, s_next);
    }
    if (ok && n_kv > 0) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(&s.o_done[(n_kv - 1) & 1], ((n_kv - 1) >> 1) & 1, a.err, kErrFwdSoftmax));
      tc_fence_after_sync();
    }
    if (ok) {
      // epilogue: O = acc / (l * keep), statistics before dropout
      const float inv = (l > 0.f) ? g.inv_keep / l : 0.f;
      const int64_t orow = q_elem(g, sq, w.b, w.n, i);
      uint32_t acc[D / 32][32];  // the row of O (fp32 bits); zero when no key is visible
      if (n_kv > 0) {
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) tmem_ld_32x32b_x32(tmem + lane_off + kColO + ch * 32, acc[ch]);
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) tmem_ld_wait(acc[ch]);  // one wait for all the loads
      } else {
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch)
#pragma unroll
          for (int t = 0; t < 32; ++t) acc[ch][t] = 0u;
      }
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        if (ch * 32 >= g.D) break;  // columns past D are padding
        float o[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) o[t] = __uint_as_float(acc[ch][t]) * inv;
        if (row_valid) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            if (ch * 32 + q4 * 8 < g.D && in_bounds(orow + ch * 32 + q4 * 8, 8, g.n_q_elems, a.err))
              store8<F16>(a.out, orow + ch * 32 + q4 * 8, &o[q4 * 8], g.out_f32);
        }
      }
      if (row_valid) {
        const int64_t si = stat_index(g, sq, w.b, w.n, i);
        const bool empty = (m_true == -INFINITY);
        if (in_bounds(si, 1, g.n_stats, a.err)) {
          a.smax[si] = empty ? -INFINITY : m_true * kLn2;
          a.ssum[si] = empty ? 0.f : l * ex2_approx(m_use - m_true);
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int DM, bool F16, int CAP>
cudaError_t launch_fwd_t(const FwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, cudaStream_t stream) {
  const size_t smem = sizeof(FwdSmem<D>) + 1024;
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t e = set_smem_limit(swa_fwd_kernel<D, DM, F16, CAP>, smem, smem_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(swa_fwd_kernel<D, DM, F16, CAP>, dim3(tab.n_items), dim3(224), smem, stream, a, tab, mq, mk, mv);
}

}  // namespace

template <int CAP>
cudaError_t launch_forward(const FwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq, const CUtensorMap& mk,
                           const CUtensorMap& mv, cudaStream_t stream) {
  if (tab.n_items == 0) return cudaSuccess;
  // (drop mode, D, element type) -> one of the twelve instantiations
  switch ((drop_mode_of(a.g.has_mask, a.g.drop_gen) * 2 + (a.g.D <= 64 ? 0 : 1)) * 2 + (a.g.f16 ? 1 : 0)) {
    case 0: return launch_fwd_t<64, 0, false>(a, tab, mq, mk, mv, stream);
    case 1: return launch_fwd_t<64, 0, true>(a, tab, mq, mk, mv, stream);
    case 2: return launch_fwd_t<128, 0, false>(a, tab, mq, mk, mv, stream);
    case 3: return launch_fwd_t<128, 0, true>(a, tab, mq, mk, mv, stream);
    case 4: return launch_fwd_t<64, 1, false>(a, tab, mq, mk, mv, stream);
    case 5: return launch_fwd_t<64, 1, true>(a, tab, mq, mk, mv, stream);
    case 6: return launch_fwd_t<128, 1, false>(a, tab, mq, mk, mv, stream);
    case 7: return launch_fwd_t<128, 1, true>(a, tab, mq, mk, mv, stream);
    case 8: return launch_fwd_t<64, 2, false>(a, tab, mq, mk, mv, stream);
    case 9: return launch_fwd_t<64, 2, true>(a, tab, mq, mk, mv, stream);
    case 10: return launch_fwd_t<128, 2, false>(a, tab, mq, mk, mv, stream);
    default: return launch_fwd_t<128, 2, true>(a, tab, mq, mk, mv, stream);
  }
}

template cudaError_t launch_forward<kSmallTable>(const FwdArgs&, const SeqTable<kSmallTable>&, const CUtensorMap&,
                                                 const CUtensorMap&, const CUtensorMap&, cudaStream_t);
template cudaError_t launch_forward<kLargeTable>(const FwdArgs&, const SeqTable<kLargeTable>&, const CUtensorMap&,
                                                 const CUtensorMap&, const CUtensorMap&, cudaStream_t);

}  // namespace swa
