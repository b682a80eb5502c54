// swa_fwd_pair.cu — sliding-window attention forward for D <= 64, two query
// tiles per CTA.
//
// The same computation as swa_fwd.cu (FlashAttentionVarLenScore doc,
// "计算公式"; the online softmax of the PyPTO-Gym article's forward), with
// one CTA covering two consecutive 128-row query tiles A = 2p and B = 2p + 1
// of one (batch, head).  At D <= 64 TMEM holds a score tile, an O
// accumulator and a P tile for each half (512 columns in all), so the halves
// run as two softmax pipelines that share the K / V loads and the tensor
// pipe.  Warps:
//   warps 0-3  softmax + epilogue of half A, one thread per query row
//   warps 4-7  the same for half B
//   warp  8    TMA producer: both Q tiles once; K and V of the union of the
//              halves' key ranges through 3-stage rings
//   warp  9    tcgen05 issuer of S_h = Q_h K^T (per key tile: A, then B)
//   warp 10    tcgen05 issuer of O_h += P_h V (P_h taken from TMEM)
// Each scheduler hosts one softmax warp of each half, so one half's
// dependency chains (the exponentials, the loads of S, the stores of P) run
// in the issue slots the other leaves idle, and one half's start-up and
// epilogue overlap the other's tiles.  Per half, S and P are single
// buffers: S_h(t+1) may be computed once the softmax holds S_h(t) in
// registers, and P_h(t+1) is stored once O_h += P_h(t) V is done.
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,320), O_B [320,384),
// P_A [384,448), P_B [448,512).
#include "swa_device.cuh"

namespace swa {
namespace {

constexpr int kPairStages = 3;
constexpr int kPairThreads = 352;

template <int D>
struct PairSmem {
  static constexpr int kTileBytes = kTileM * D * 2;
  alignas(1024) uint8_t q[2][kTileBytes];
  alignas(1024) uint8_t k[kPairStages][kTileBytes];
  alignas(1024) uint8_t v[kPairStages][kTileBytes];
  uint64_t q_full, k_full[kPairStages], v_full[kPairStages], k_empty[kPairStages], v_empty[kPairStages];
  uint64_t s_full[2], s_free[2], p_full[2], o_done[2];  // per half
  uint64_t drain_s, drain_pv;
  uint64_t never;  // completed by nothing: the target of the stall test hook
  uint32_t tmem_base;
};
static_assert(sizeof(PairSmem<64>) + 1024 <= 232448, "shared memory budget");

constexpr uint32_t kPairTmemCols = 512;
__device__ __forceinline__ uint32_t col_s(int h) { return static_cast<uint32_t>(h) * 128u; }
__device__ __forceinline__ uint32_t col_o(int h) { return 256u + static_cast<uint32_t>(h) * 64u; }
__device__ __forceinline__ uint32_t col_p(int h) { return 384u + static_cast<uint32_t>(h) * 64u; }
constexpr float kPairLn2 = 0.6931471805599453f;
// Rescale O only when the running max grows by more than 2^8 (log2 units).
constexpr float kPairRescale = 8.0f;

// The key tiles [t0, t0 + n) of query tile qt, or none if the tile does not exist.
struct HalfRange {
  int t0, n;
};
__device__ __forceinline__ HalfRange half_range(const Geometry& g, const SeqInfo& s, int qt) {
  HalfRange r{0, 0};
  if (qt * kTileM < s.q_len) key_tiles_of_query_tile(g, s, qt, &r.t0, &r.n);
  return r;
}

template <int D, int DM, bool F16, int CAP>
__global__ void __launch_bounds__(kPairThreads, 1)
    swa_fwd_pair_kernel(const FwdArgs a, const __grid_constant__ SeqTable<CAP> tab,
                        const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                        const __grid_constant__ CUtensorMap mv) {
  extern __shared__ uint8_t smem_raw[];
  PairSmem<D>& s = *reinterpret_cast<PairSmem<D>*>(align1024(smem_raw));
  constexpr int kTileBytes = PairSmem<D>::kTileBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // q, k, v, the outputs and the status word may belong to the previous grid
  // on the stream (this kernel is launched with programmatic serialization):
  // wait for it before touching any of them.  No early trigger: the next
  // grid starts when this one ends (backward CTAs made resident during the
  // forward's last wave slowed the whole step)
  griddep_wait();
  if (a.clear_err && blockIdx.x == 0 && threadIdx.x == 0) *a.err = 0;
  const Geometry& g = a.g;
  const Item w = resolve_item(tab, a.g, static_cast<int>(blockIdx.x), a.g.N);  // w.tile: the pair p
  const int hk = w.n / a.g.group;  // the key/value head this query head reads
  const SeqInfo sq = w.s;
  const HalfRange ra = half_range(g, sq, 2 * w.tile), rb = half_range(g, sq, 2 * w.tile + 1);
  const bool has_b = (2 * w.tile + 1) * kTileM < sq.q_len;
  // the key tiles either half visits: [u0, u0 + n_u)
  int u0, n_u;
  key_tiles_of_query_pair(g, sq, w.tile, &u0, &n_u);
  auto uses = [&](int h, int j) {
    const HalfRange& r = h ? rb : ra;
    return j >= r.t0 && j < r.t0 + r.n;
  };

  // The producer's lane initialises the barriers and issues the loads of
  // both Q tiles and the first K tile before the CTA-wide barrier.
  if (warp == 8 && lane == 0) {
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < kPairStages; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
      mbar_init(&s.v_empty[i], 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&s.s_full[h], 1);
      mbar_init(&s.s_free[h], kTileM);
      mbar_init(&s.p_full[h], kTileM);
      mbar_init(&s.o_done[h], 1);
    }
    mbar_init(&s.drain_s, 1);
    mbar_init(&s.drain_pv, 1);
    mbar_init(&s.never, 1);
    fence_mbar_init();
    if (n_u > 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
      mbar_arrive_expect_tx(&s.q_full, (has_b ? 2 : 1) * kTileBytes);
      tma_rows<D>(s.q[0], &mq, &s.q_full, g, w.b, w.n, sq.q_start, 2 * w.tile * kTileM);
      if (has_b) tma_rows<D>(s.q[1], &mq, &s.q_full, g, w.b, w.n, sq.q_start, (2 * w.tile + 1) * kTileM);
      mbar_arrive_expect_tx(&s.k_full[0], kTileBytes);
      tma_rows<D>(s.k[0], &mk, &s.k_full[0], g, w.b, hk, sq.kv_start, u0 * kTileN);
    }
  }
  if (warp == 9) {
    tmem_alloc(&s.tmem_base, kPairTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s.tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0 && n_u > 0) {
      int k_issued = 1, v_issued = 0;  // K(0) went out before the CTA-wide barrier
      for (int it = 0; it < n_u; ++it) {
        const int st = it % kPairStages;
        const uint32_t use = it / kPairStages;
        const int j0 = (u0 + it) * kTileN;
        if (it > 0) {
          if (it >= kPairStages && !mbar_wait(&s.k_empty[st], (use - 1) & 1, a.err, kErrFwdLoad)) break;
          mbar_arrive_expect_tx(&s.k_full[st], kTileBytes);
          tma_rows<D>(s.k[st], &mk, &s.k_full[st], g, w.b, hk, sq.kv_start, j0);
          ++k_issued;
        }
        if (it >= kPairStages && !mbar_wait(&s.v_empty[st], (use - 1) & 1, a.err, kErrFwdLoad)) break;
        mbar_arrive_expect_tx(&s.v_full[st], kTileBytes);
        tma_rows<D>(s.v[st], &mv, &s.v_full[st], g, w.b, hk, sq.kv_start, j0);
        ++v_issued;
      }
      // every copy issued has landed before the CTA may exit
      mbar_wait_drain(&s.q_full, 0);
      for (int st = 0; st < kPairStages; ++st) {
        const int uk = (k_issued - st + kPairStages - 1) / kPairStages;
        const int uv = (v_issued - st + kPairStages - 1) / kPairStages;
        if (uk > 0) mbar_wait_drain(&s.k_full[st], (uk - 1) & 1);
        if (uv > 0) mbar_wait_drain(&s.v_full[st], (uv - 1) & 1);
      }
    }
  } else if (warp == 9) {
    // ----------------------------------------------- S_h = Q_h K^T issuer --
    if (lane == 0 && n_u > 0) {
      constexpr uint32_t kIdS = idesc_f16_f32(kTileM, kTileN, false, false, F16);
      const int nk = d_steps(g);
      int issued[2] = {0, 0};  // S tiles issued per half
      bool ok = mbar_wait(&s.q_full, 0, a.err, kErrFwdMma);
      for (int it = 0; ok && it < n_u; ++it) {
        const int st = it % kPairStages, j = u0 + it;
        if (!mbar_wait(&s.k_full[st], (it / kPairStages) & 1, a.err, kErrFwdMma)) break;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!uses(h, j)) continue;
          // single S buffer: the softmax of half h holds S_h(c - 1) in registers
          const int c = issued[h];
          if (c >= 1 && !mbar_wait(&s.s_free[h], (c - 1) & 1, a.err, kErrFwdMma)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t dq_ = sdesc_sw128(smem_u32(s.q[h]), 16, 1024);
          const uint64_t dk_ = sdesc_sw128(smem_u32(s.k[st]), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            if (kk >= nk) break;
            const uint32_t off = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
            umma_bf16_ss(tmem + col_s(h), sdesc_advance(dq_, off), sdesc_advance(dk_, off), kIdS, kk > 0);
          }
          umma_commit(&s.s_full[h]);
          issued[h] = c + 1;
        }
        if (!ok) break;
        umma_commit(&s.k_empty[st]);
      }
      umma_commit(&s.drain_s);
      mbar_wait_drain(&s.drain_s, 0);
    }
  } else if (warp == 10) {
    // -------------------------------------------------- O_h += P_h V issuer --
    if (lane == 0 && n_u > 0) {
      constexpr uint32_t kIdO = idesc_f16_f32(kTileM, D, false, true, F16);
      int issued[2] = {0, 0};  // PV tiles issued per half
      bool ok = true;
      for (int it = 0; ok && it < n_u; ++it) {
        const int st = it % kPairStages, j = u0 + it;
        if (!mbar_wait(&s.v_full[st], (it / kPairStages) & 1, a.err, kErrFwdMma)) break;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!uses(h, j)) continue;
          const int c = issued[h];
          if (!mbar_wait(&s.p_full[h], c & 1, a.err, kErrFwdMma)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t dv_ = sdesc_sw128(smem_u32(s.v[st]), kAtomBytes, 1024);
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk)  // O_h += P_h V  (A = P_h in TMEM)
            umma_bf16_ts(tmem + col_o(h), tmem + col_p(h) + kk * 8, sdesc_advance(dv_, kk * 2048), kIdO,
                         (c > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&s.o_done[h]);
          issued[h] = c + 1;
        }
        if (!ok) break;
        umma_commit(&s.v_empty[st]);
      }
      umma_commit(&s.drain_pv);
      mbar_wait_drain(&s.drain_pv, 0);
    }
  } else {
    // ---------------------------------- softmax + epilogue of one half --
    const int h = warp >> 2;  // 0: half A, 1: half B
    const HalfRange rh = h ? rb : ra;
    const int n_kv = rh.n, kv_t0 = rh.t0;
    const int q0 = (2 * w.tile + h) * kTileM;
    const int r = (warp & 3) * 32 + lane;  // TMEM lane == row of the half's tile
    const int i = q0 + r;
    const bool row_valid = i < sq.q_len;
    int wlo, whi;
    key_window(g, sq, i, wlo, whi);
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c = g.scale_log2;
    float m_use = -INFINITY, m_true = -INFINITY, l = 0.f;
    bool ok = true;
    // test hook: wait on a barrier that nothing completes, so the bounded
    // wait runs out and the launch reports it
    if (g.stall & kStallForward)
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(&s.never, 0, a.err, kErrFwdSoftmax));
    for (int it = 0; ok && it < n_kv; ++it) {
      // This tile's keep bits, loaded at the start of the tile: the other
      // half's warps cover the load latency, and fetching them a tile ahead
      // (as the one-tile kernel does) cost more in spilled registers than it
      // saved here (0.0706 vs 0.0734-0.0745 ms on BNSD 4x16x2048x64).
      uint32_t bits[4] = {~0u, ~0u, ~0u, ~0u};
      if (DM == 1) {
        bits[0] = bits[1] = bits[2] = bits[3] = 0u;
        if (row_valid) load_keep_bits(a.mask, sq, w.n, i, (kv_t0 + it) * kTileN, bits, g.n_mask_bytes, a.err);
      }
      // warp-uniform outcome: the tcgen05.ld below is warp-collective
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&s.s_full[h], it & 1, a.err, kErrFwdSoftmax))) {
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
        const uint32_t base = tmem + lane_off + col_s(h);
        tmem_ld_32x32b_x32(base + 0, x0);
        tmem_ld_32x32b_x32(base + 32, x1);
        tmem_ld_32x32b_x32(base + 64, x2);
        tmem_ld_32x32b_x32(base + 96, x3);
        tmem_ld_wait(x0);
        tmem_ld_wait(x1);
        tmem_ld_wait(x2);
        tmem_ld_wait(x3);
      }
      tc_fence_before_sync();
      mbar_arrive(&s.s_free[h]);  // S_h(it + 1) may now be computed over S_h(it)
      // O_h += P_h(it - 1) V must be done before P_h(it) goes into the single
      // P buffer (and before O_h is rescaled): probe now, use the answer
      // after the exponentials
      const bool pv_done = it < 1 || mbar_test(&s.o_done[h], (it - 1) & 1);
      auto X = [&](int t) -> float { return __uint_as_float(xr[t]); };

      const int j0 = (kv_t0 + it) * kTileN;
      // Positive scale: maximum on the raw scores, the scale folded into one
      // packed FMA per pair, p = exp2(x*c - m); keys outside the window
      // (partial tiles only) become -inf first.  A scale <= 0 takes scale,
      // mask, exp2(x - m).
      const bool fold = c > 0.f;
      const bool fast = fold && tile_fully_visible(g, sq, q0, j0);
      float mx;
      {
        float m8[8];  // eight independent partial maxima
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
      const bool need = m_new > m_use + kPairRescale;
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
      if (!__all_sync(0xFFFFFFFFu, pv_done) &&
          !__all_sync(0xFFFFFFFFu, mbar_wait(&s.o_done[h], (it - 1) & 1, a.err, kErrFwdSoftmax))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      if (it >= 1 && warp_need) {  // no P V of this half is in flight now
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t t32[32];
          const uint32_t addr = tmem + lane_off + col_o(h) + ch * 32;
          tmem_ld_32x32b_x32(addr, t32);
          tmem_ld_wait(t32);
#pragma unroll
          for (int t = 0; t < 32; ++t) t32[t] = __float_as_uint(__uint_as_float(t32[t]) * alpha);
          tmem_st_32x32b_x32(addr, t32);
        }
      }
      tmem_st_32x32b_x32(tmem + lane_off + col_p(h), *reinterpret_cast<const uint32_t(*)[32]>(&xr[0]));
      tmem_st_32x32b_x32(tmem + lane_off + col_p(h) + 32, *reinterpret_cast<const uint32_t(*)[32]>(&xr[32]));
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&s.p_full[h]);
    }
    if (ok && n_kv > 0) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(&s.o_done[h], (n_kv - 1) & 1, a.err, kErrFwdSoftmax));
      tc_fence_after_sync();
    }
    if (ok && q0 < sq.q_len) {
      // epilogue: O = acc / (l * keep), statistics before dropout
      const float inv = (l > 0.f) ? g.inv_keep / l : 0.f;
      const int64_t orow = q_elem(g, sq, w.b, w.n, i);
      uint32_t acc[D / 32][32];  // the row of O (fp32 bits); zero when no key is visible
      if (n_kv > 0) {
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) tmem_ld_32x32b_x32(tmem + lane_off + col_o(h) + ch * 32, acc[ch]);
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) tmem_ld_wait(acc[ch]);
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
          a.smax[si] = empty ? -INFINITY : m_true * kPairLn2;
          a.ssum[si] = empty ? 0.f : l * ex2_approx(m_use - m_true);
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kPairTmemCols);
  }
}

template <int DM, bool F16, int CAP>
cudaError_t launch_fwd_pair_t(const FwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq,
                              const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t stream) {
  const size_t smem = sizeof(PairSmem<64>) + 1024;
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t e = set_smem_limit(swa_fwd_pair_kernel<64, DM, F16, CAP>, smem, smem_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(swa_fwd_pair_kernel<64, DM, F16, CAP>, dim3(tab.n_items), dim3(kPairThreads), smem, stream, a,
                    tab, mq, mk, mv);
}

}  // namespace

// D <= 64 only; the table's entries count query tile pairs (tiles = ceil(query tiles / 2)).
template <int CAP>
cudaError_t launch_forward_pair(const FwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq,
                                const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t stream) {
  if (tab.n_items == 0) return cudaSuccess;
  switch (drop_mode_of(a.g.has_mask, a.g.drop_gen) * 2 + (a.g.f16 ? 1 : 0)) {
    case 0: return launch_fwd_pair_t<0, false>(a, tab, mq, mk, mv, stream);
    case 1: return launch_fwd_pair_t<0, true>(a, tab, mq, mk, mv, stream);
    case 2: return launch_fwd_pair_t<1, false>(a, tab, mq, mk, mv, stream);
    case 3: return launch_fwd_pair_t<1, true>(a, tab, mq, mk, mv, stream);
    case 4: return launch_fwd_pair_t<2, false>(a, tab, mq, mk, mv, stream);
    default: return launch_fwd_pair_t<2, true>(a, tab, mq, mk, mv, stream);
  }
}

template cudaError_t launch_forward_pair<kSmallTable>(const FwdArgs&, const SeqTable<kSmallTable>&,
                                                      const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                      cudaStream_t);
template cudaError_t launch_forward_pair<kLargeTable>(const FwdArgs&, const SeqTable<kLargeTable>&,
                                                      const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                      cudaStream_t);

}  // namespace swa
