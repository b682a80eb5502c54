// swa_bwd_dq.cu — sliding-window attention backward, query-major pass: dQ.
//
// Per (query tile i, key tile j) pair inside the BAND (PyPTO-Gym article,
// "反向公式", the dQ row of the formulas):
//   S  = Q K^T,  P = exp2(S*scale*log2e - lse2),  dP = dY V^T,
//   dS = P * (dP * z/keep - D),  dQ += dS K,  dQ = scale * dQ at the end.
// With dropout the tiles carry P * (z*dP - keep*D), 1/keep times dS, and the
// epilogue multiplies by scale/keep instead.
// dQ accumulates in TMEM over the key tiles of the band and is written once:
// no accumulation through global memory (the measured fp32 reduce-add ceiling
// of the L2 would otherwise bound the backward), and the result is
// deterministic.
//
// One CTA = one 128-row query tile of one (batch, head).  Warps:
//   warps 0-7  compute: warp w owns TMEM lanes 32*(w%4).. (query rows) and key
//              columns 64*(w/4).. of each tile; in the epilogue, dQ columns
//              [w/4 * D/2, +D/2)
//   warp  8    TMA producer: Q, dY once; K through a 3-stage ring (a K tile
//              is read by S and, last, by dQ) and V through a 2-stage ring
//              (read by dP only, so it is released early)
//   warp  9    tcgen05 issuer of S (SS)
//   warp 10    tcgen05 issuer of dQ += dS K (TS)
//   warp 11    tcgen05 issuer of dP (SS)
// One issuing thread per GEMM stream: the tensor pipe's queue is shallow, so
// a thread issuing one GEMM blocks until most of it has run, and a GEMM whose
// inputs are ready must not wait behind another GEMM's issue (with S and dP
// on one thread, S(j+1) sat ~700 cycles behind dP(j)).
// TMEM columns: S [0,128), dP [128,256), dQ [256,256+D), and two bf16 dS
// buffers [384,448), [448,512) that the dQ MMA reads as its A operand.
// S(j+1) is issued as soon as the compute warps hold S(j) in registers and
// dP(j+1) as soon as they hold dP(j), so both are ready before the compute
// warps reach them; dQ(j) follows dS(j).
#include "swa_device.cuh"

namespace swa {
namespace {

template <int D>
struct DqSmem {
  static constexpr int kTileBytes = kTileM * D * 2;
  alignas(1024) uint8_t q[kTileBytes];
  alignas(1024) uint8_t dy[kTileBytes];
  alignas(1024) uint8_t k[3][kTileBytes];
  alignas(1024) uint8_t v[2][kTileBytes];
  uint64_t qdy_full, k_full[3], k_empty[3], v_full[2], v_empty[2];
  uint64_t s_full, s_loaded, dp_full, dp_loaded, ds_full[2], ds_free[2], drain_s, drain_dp, drain_dq;
  uint64_t never;  // completed by nothing: the target of the stall test hook
  uint32_t tmem_base;
};
static_assert(sizeof(DqSmem<128>) + 1024 <= 232448, "shared memory budget");

constexpr int kThreads = 384;
constexpr int kComputeThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 384;  // dS buffer b at kColDS + 64*b

// Warp-uniform bounded wait of the compute warps.  A warp vote (not a
// CTA-wide barrier) keeps each warp converged for its warp-collective TMEM
// accesses; no compute step reads what another warp wrote in TMEM.
__device__ __forceinline__ bool compute_wait(uint64_t* bar, uint32_t parity, int* err) {
  return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, err, kErrBwdCompute));
}

template <int D, int DM, bool F16, int CAP>
__global__ void __launch_bounds__(kThreads, 1)
    swa_bwd_dq_kernel(const BwdArgs a, const __grid_constant__ SeqTable<CAP> tab, const __grid_constant__ CUtensorMap mq,
                      const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                      const __grid_constant__ CUtensorMap mdy) {
  extern __shared__ uint8_t smem_raw[];
  DqSmem<D>& s = *reinterpret_cast<DqSmem<D>*>(align1024(smem_raw));
  constexpr int kTileBytes = DqSmem<D>::kTileBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_launch_dependents();
  const Geometry& g = a.g;
  const Item w = resolve_item(tab, a.g, static_cast<int>(blockIdx.x), a.g.N);
  const int hk = w.n / a.g.group;  // the key/value head this query head reads
  const SeqInfo sq = w.s;
  const int q0 = w.tile * kTileM;

  // key tiles touched by this query tile
  int kv_t0, n_kv;
  key_tiles_of_query_tile(g, sq, w.tile, &kv_t0, &n_kv);

  // The producer's lane initialises the barriers and issues the loads of Q,
  // dY and the first K and V tiles before the CTA-wide barrier, so their
  // latency runs while TMEM is allocated.
  if (warp == 8 && lane == 0) {
    mbar_init(&s.qdy_full, 1);
    for (int b = 0; b < 3; ++b) {
      mbar_init(&s.k_full[b], 1);
      mbar_init(&s.k_empty[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s.v_full[b], 1);
      mbar_init(&s.v_empty[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s.ds_full[b], kComputeThreads);
      mbar_init(&s.ds_free[b], 1);
    }
    mbar_init(&s.s_full, 1);
    mbar_init(&s.s_loaded, kComputeThreads);
    mbar_init(&s.dp_full, 1);
    mbar_init(&s.dp_loaded, kComputeThreads);
    mbar_init(&s.drain_s, 1);
    mbar_init(&s.drain_dp, 1);
    mbar_init(&s.drain_dq, 1);
    mbar_init(&s.never, 1);
    fence_mbar_init();
    if (n_kv > 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
      tma_prefetch_desc(&mdy);
      mbar_arrive_expect_tx(&s.qdy_full, 2 * kTileBytes);
      tma_rows<D>(s.q, &mq, &s.qdy_full, g, w.b, w.n, sq.q_start, q0);
      tma_rows<D>(s.dy, &mdy, &s.qdy_full, g, w.b, w.n, sq.q_start, q0);
      mbar_arrive_expect_tx(&s.k_full[0], kTileBytes);
      tma_rows<D>(s.k[0], &mk, &s.k_full[0], g, w.b, hk, sq.kv_start, kv_t0 * kTileN);
      mbar_arrive_expect_tx(&s.v_full[0], kTileBytes);
      tma_rows<D>(s.v[0], &mv, &s.v_full[0], g, w.b, hk, sq.kv_start, kv_t0 * kTileN);
    }
  }
  if (warp == 9) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s.tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0 && n_kv > 0) {
      int k_issued = 1, v_issued = 1;  // Q, dY, K(0) and V(0) went out before the CTA-wide barrier
      for (int j = 1; j < n_kv; ++j) {
        const int jr = (kv_t0 + j) * kTileN;
        const int kb = j % 3, vb = j & 1;
        // K(j) reuses the stage of K(j-3), free once dQ(j-3) is done
        if (j >= 3 && !mbar_wait(&s.k_empty[kb], ((j / 3) - 1) & 1, a.err, kErrBwdLoad)) break;
        mbar_arrive_expect_tx(&s.k_full[kb], kTileBytes);
        tma_rows<D>(s.k[kb], &mk, &s.k_full[kb], g, w.b, hk, sq.kv_start, jr);
        ++k_issued;
        // V(j) reuses the stage of V(j-2), free once dP(j-2) is done
        if (j >= 2 && !mbar_wait(&s.v_empty[vb], ((j >> 1) - 1) & 1, a.err, kErrBwdLoad)) break;
        mbar_arrive_expect_tx(&s.v_full[vb], kTileBytes);
        tma_rows<D>(s.v[vb], &mv, &s.v_full[vb], g, w.b, hk, sq.kv_start, jr);
        ++v_issued;
      }
      // every copy issued has landed before the CTA may exit
      mbar_wait_drain(&s.qdy_full, 0);
      for (int b = 0; b < 3; ++b) {
        const int uses = (k_issued - b + 2) / 3;
        if (uses > 0) mbar_wait_drain(&s.k_full[b], (uses - 1) & 1);
      }
      for (int b = 0; b < 2; ++b) {
        const int uses = (v_issued - b + 1) / 2;
        if (uses > 0) mbar_wait_drain(&s.v_full[b], (uses - 1) & 1);
      }
    }
  } else if (warp == 9 || warp == 11) {
    // ------------------------------------------ tcgen05 issuers of S, dP --
    if (lane == 0 && n_kv > 0) {
      constexpr uint32_t kIdS = idesc_f16_f32(kTileM, kTileN, false, false, F16);  // S, dP
      const uint32_t q_addr = smem_u32(s.q), dy_addr = smem_u32(s.dy);
      const int nk = d_steps(g);
      if (warp == 9) {
        // S(j) = Q K_j^T; S(j+1) once the compute warps hold S(j) in registers
        for (int j = 0; j < n_kv; ++j) {
          if (j == 0 && !mbar_wait(&s.qdy_full, 0, a.err, kErrBwdMma)) break;
          if (j > 0 && !mbar_wait(&s.s_loaded, (j - 1) & 1, a.err, kErrBwdMma)) break;
          if (!mbar_wait(&s.k_full[j % 3], (j / 3) & 1, a.err, kErrBwdMma)) break;
          tc_fence_after_sync();
          const uint64_t dq_ = sdesc_sw128(q_addr, 16, 1024), dk_ = sdesc_sw128(smem_u32(s.k[j % 3]), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            if (kk >= nk) break;
            const uint32_t off = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
            umma_bf16_ss(tmem + kColS, sdesc_advance(dq_, off), sdesc_advance(dk_, off), kIdS, kk > 0);
          }
          umma_commit(&s.s_full);
        }
        umma_commit(&s.drain_s);
        mbar_wait_drain(&s.drain_s, 0);
      } else {
        // dP(j) = dY V_j^T; dP(j+1) once the compute warps hold dP(j)
        for (int j = 0; j < n_kv; ++j) {
          if (j == 0 && !mbar_wait(&s.qdy_full, 0, a.err, kErrBwdMma)) break;
          if (j > 0 && !mbar_wait(&s.dp_loaded, (j - 1) & 1, a.err, kErrBwdMma)) break;
          if (!mbar_wait(&s.v_full[j & 1], (j >> 1) & 1, a.err, kErrBwdMma)) break;
          tc_fence_after_sync();
          const uint64_t ddy = sdesc_sw128(dy_addr, 16, 1024), dv_ = sdesc_sw128(smem_u32(s.v[j & 1]), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            if (kk >= nk) break;
            const uint32_t off = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
            umma_bf16_ss(tmem + kColDP, sdesc_advance(ddy, off), sdesc_advance(dv_, off), kIdS, kk > 0);
          }
          umma_commit(&s.dp_full);
          umma_commit(&s.v_empty[j & 1]);
        }
        umma_commit(&s.drain_dp);
        mbar_wait_drain(&s.drain_dp, 0);
      }
    }
  } else if (warp == 10) {
    // ------------------------------------------------ dQ += dS K issuer --
    if (lane == 0 && n_kv > 0) {
      constexpr uint32_t kIdQ = idesc_f16_f32(kTileM, D, false, true, F16);
      for (int j = 0; j < n_kv; ++j) {
        const int b = j & 1;
        if (!mbar_wait(&s.ds_full[b], (j >> 1) & 1, a.err, kErrBwdMma)) break;
        tc_fence_after_sync();
        const uint64_t dk_ = sdesc_sw128(smem_u32(s.k[j % 3]), kAtomBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk)  // dQ += dS(j) K_j  (A = dS in TMEM, K dim = keys)
          umma_bf16_ts(tmem + kColDQ, tmem + kColDS + b * 64 + kk * 8, sdesc_advance(dk_, kk * 2048), kIdQ,
                       (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&s.ds_free[b]);
        // K(j) was also read by S(j), which finished before dS(j) existed
        umma_commit(&s.k_empty[j % 3]);
      }
      umma_commit(&s.drain_dq);
      mbar_wait_drain(&s.drain_dq, 0);
    }
  } else {
    // ------------------------------------------- compute warps (0..7) -----
    const int wq = warp & 3, h = warp >> 2;  // lane quarter, key-column half
    const int r = wq * 32 + lane;            // TMEM lane = query row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int cbase = h * 64;
    const float c = g.scale_log2;
    const int i = q0 + r;
    const bool row_valid = i < sq.q_len;
    int wlo, whi;
    key_window(g, sq, i, wlo, whi);
    griddep_wait();  // lse2 and D come from the preprocess grid, which ran before the previous grid ended
    float lse2 = INFINITY, drow = 0.f;
    if (row_valid) {
      const int64_t si = ws_stat_index(g, sq, w.b, w.n, i);
      if (in_bounds(si, 1, g.n_stats, a.err)) {
        lse2 = a.lse2[si];
        drow = a.dsum[si];
      }
      if constexpr (DM != 0) drow *= g.keep;  // the loop forms P * (z dP - keep D)
    }
    // keep bits of this thread's 64 key columns of key tile j (two words)
    auto fetch_bits = [&](int j, uint32_t& kb0, uint32_t& kb1) {
      kb0 = kb1 = 0xFFFFFFFFu;
      if (DM == 1 && row_valid) {
        uint32_t bits[4];
        load_keep_bits(a.mask, sq, w.n, i, (kv_t0 + j) * kTileN, bits, g.n_mask_bytes, a.err);
        kb0 = h ? bits[2] : bits[0];
        kb1 = h ? bits[3] : bits[1];
      } else if (DM == 2) {
        uint32_t bits[2];
        gen_keep_words<2>(g, stat_index(g, sq, w.b, w.n, i), ((kv_t0 + j) * kTileN + cbase) >> 4, bits);
        kb0 = bits[0];
        kb1 = bits[1];
      }
    };
    uint32_t n_kb0 = 0xFFFFFFFFu, n_kb1 = 0xFFFFFFFFu;
    if (DM != 0 && n_kv > 0) fetch_bits(0, n_kb0, n_kb1);
    bool ok = true;
    // test hook: wait on a barrier that nothing completes, so the bounded
    // wait runs out and the launch reports it
    if (g.stall & kStallQueryMajor) ok = compute_wait(&s.never, 0, a.err);
    for (int j = 0; ok && j < n_kv; ++j) {
      const int b = j & 1;
      const uint32_t u = (j >> 1) & 1;
      const uint32_t kb0 = n_kb0, kb1 = n_kb1;
      if (DM != 0 && j + 1 < n_kv) fetch_bits(j + 1, n_kb0, n_kb1);
      const int jb = (kv_t0 + j) * kTileN;
      const bool full = tile_fully_visible(g, sq, q0, jb);

      // ---- S -> P (kept in registers)
      if (!compute_wait(&s.s_full, j & 1, a.err)) { ok = false; break; }
      tc_fence_after_sync();
      float p[64];
      {
        uint32_t s0[32], s1[32];
        tmem_ld_32x32b_x32(tmem + lane_off + kColS + cbase, s0);
        tmem_ld_32x32b_x32(tmem + lane_off + kColS + cbase + 32, s1);
        tmem_ld_wait(s0);
        tmem_ld_wait(s1);
        tc_fence_before_sync();
        mbar_arrive(&s.s_loaded);
        // Two copies of the loop: tiles entirely inside the window (nearly
        // all of them) need no per-element mask.  In the masked copy the
        // exp2 is unconditional and the comparisons use non-short-circuit
        // operators, so the mask compiles to selects, not branches.
        if (full) {
#pragma unroll
          for (int t = 0; t < 64; t += 2) {  // packed pairs: (s*c - lse2) in one f32x2 FMA
            float x0, x1;
            ffma2_bcast(x0, x1, __uint_as_float(t < 32 ? s0[t] : s1[t - 32]),
                        __uint_as_float(t + 1 < 32 ? s0[t + 1] : s1[t - 31]), c, -lse2);
            p[t] = ex2_approx(x0);
            p[t + 1] = ex2_approx(x1);
          }
        } else {
          const int lo_t = wlo - (jb + cbase), hi_t = whi - (jb + cbase);  // visible t in [lo_t, hi_t]
#pragma unroll
          for (int t = 0; t < 64; ++t) {
            const float e = ex2_approx(__uint_as_float(t < 32 ? s0[t] : s1[t - 32]) * c - lse2);
            p[t] = ((t >= lo_t) & (t <= hi_t)) ? e : 0.f;
          }
        }
      }
      // ---- dP -> dS (packed bf16)
      if (!compute_wait(&s.dp_full, j & 1, a.err)) { ok = false; break; }
      tc_fence_after_sync();
      uint32_t dk[32];
      {
        uint32_t d0[32], d1[32];
        tmem_ld_32x32b_x32(tmem + lane_off + kColDP + cbase, d0);
        tmem_ld_32x32b_x32(tmem + lane_off + kColDP + cbase + 32, d1);
        tmem_ld_wait(d0);
        tmem_ld_wait(d1);
        tc_fence_before_sync();
        mbar_arrive(&s.dp_loaded);
        // dS = P * (dP - D), packed pairs; with dropout P * (z dP - keep D),
        // 1/keep times dS, the epilogue taking the 1/keep
#pragma unroll
        for (int t2 = 0; t2 < 32; ++t2) {
          const int t = 2 * t2;
          float dp0 = __uint_as_float(t < 32 ? d0[t] : d1[t - 32]);
          float dp1 = __uint_as_float(t + 1 < 32 ? d0[t + 1] : d1[t - 31]);
          if (DM != 0) {
            dp0 = (((t < 32 ? kb0 : kb1) >> (t & 31)) & 1u) ? dp0 : 0.f;
            dp1 = (((t + 1 < 32 ? kb0 : kb1) >> ((t + 1) & 31)) & 1u) ? dp1 : 0.f;
          }
          float dv[2];
          fmulsub2(dv[0], dv[1], p[t], p[t + 1], dp0, dp1, drow, drow);
          dk[t2] = pack2<F16>(dv[0], dv[1]);
        }
      }
      // ---- dS -> TMEM buffer b (after dQ(j-2) has read it)
      if (j >= 2 && !compute_wait(&s.ds_free[b], u ^ 1, a.err)) { ok = false; break; }
      tmem_st_32x32b_x32(tmem + lane_off + kColDS + b * 64 + h * 32, dk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&s.ds_full[b]);
    }
    if (ok && n_kv > 0) ok = compute_wait(&s.ds_free[(n_kv - 1) & 1], ((n_kv - 1) >> 1) & 1, a.err);  // every MMA done
    // The eight compute warps agree on whether to write the epilogue: its
    // staging barrier below must see all eight or none.
    ok = named_barrier_and(1, kComputeThreads, ok);
    if (ok) {
      tc_fence_after_sync();
      // epilogue: dQ = scale / keep * acc, row r, columns [h*D/2, h*D/2 + D/2)
      const float mul = g.scale * g.inv_keep;
      constexpr int kCols = D / 2;
      const int64_t dst = q_elem(g, sq, w.b, w.n, i) + h * kCols;
#pragma unroll
      for (int ch = 0; ch < kCols / 32; ++ch) {
        if (h * kCols + ch * 32 >= g.D) break;  // columns past D are padding
        float o[32];
        if (n_kv > 0) {
          uint32_t t32[32];
          tmem_ld_32x32b_x32(tmem + lane_off + kColDQ + h * kCols + ch * 32, t32);
          tmem_ld_wait(t32);
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = __uint_as_float(t32[t]) * mul;
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = 0.f;
        }
        if (g.out_f32) {
          if (row_valid) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              if (h * kCols + ch * 32 + q4 * 8 < g.D && in_bounds(dst + ch * 32 + q4 * 8, 8, g.n_q_elems, a.err))
                store8<F16>(a.dq, dst + ch * 32 + q4 * 8, &o[q4 * 8], true);
          }
        } else {
          // staged in the Q buffer (every S is done) for whole-row stores below
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            if (h * kCols + ch * 32 + q4 * 8 < g.D)
              st_chunk_sw128(s.q, r, (h * kCols + ch * 32) / 8 + q4, pack8<F16>(&o[q4 * 8]));
        }
      }
      if (!g.out_f32) {
        // each warp store writes whole rows (one row per thread would touch
        // 32 rows, 32 cache lines, per store)
        named_barrier_sync(1, kComputeThreads);
        constexpr int kChunks = D / 8;
        constexpr int kRowsPerStore = 32 / kChunks;
        const int c = lane % kChunks;
        for (int rr = warp * kRowsPerStore + lane / kChunks; rr < kTileM; rr += 8 * kRowsPerStore) {
          const int gi = q0 + rr;
          if (gi < sq.q_len && c * 8 < g.D && in_bounds(q_elem(g, sq, w.b, w.n, gi) + c * 8, 8, g.n_q_elems, a.err))
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dq) + q_elem(g, sq, w.b, w.n, gi) + c * 8) =
                ld_chunk_sw128(s.q, rr, c);
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int DM, bool F16, int CAP>
cudaError_t launch_dq_t(const BwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq, const CUtensorMap& mk,
                        const CUtensorMap& mv, const CUtensorMap& mdy, cudaStream_t stream) {
  const size_t smem = sizeof(DqSmem<D>) + 1024;
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t e = set_smem_limit(swa_bwd_dq_kernel<D, DM, F16, CAP>, smem, smem_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(swa_bwd_dq_kernel<D, DM, F16, CAP>, dim3(tab.n_items), dim3(kThreads), smem, stream, a, tab, mq,
                    mk, mv, mdy);
}

}  // namespace

template <int CAP>
cudaError_t launch_backward_dq(const BwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq,
                               const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdy,
                               cudaStream_t stream) {
  if (tab.n_items == 0) return cudaSuccess;
  // (drop mode, D, element type) -> one of the twelve instantiations
  switch ((drop_mode_of(a.g.has_mask, a.g.drop_gen) * 2 + (a.g.D <= 64 ? 0 : 1)) * 2 + (a.g.f16 ? 1 : 0)) {
    case 0: return launch_dq_t<64, 0, false>(a, tab, mq, mk, mv, mdy, stream);
    case 1: return launch_dq_t<64, 0, true>(a, tab, mq, mk, mv, mdy, stream);
    case 2: return launch_dq_t<128, 0, false>(a, tab, mq, mk, mv, mdy, stream);
    case 3: return launch_dq_t<128, 0, true>(a, tab, mq, mk, mv, mdy, stream);
    case 4: return launch_dq_t<64, 1, false>(a, tab, mq, mk, mv, mdy, stream);
    case 5: return launch_dq_t<64, 1, true>(a, tab, mq, mk, mv, mdy, stream);
    case 6: return launch_dq_t<128, 1, false>(a, tab, mq, mk, mv, mdy, stream);
    case 7: return launch_dq_t<128, 1, true>(a, tab, mq, mk, mv, mdy, stream);
    case 8: return launch_dq_t<64, 2, false>(a, tab, mq, mk, mv, mdy, stream);
    case 9: return launch_dq_t<64, 2, true>(a, tab, mq, mk, mv, mdy, stream);
    case 10: return launch_dq_t<128, 2, false>(a, tab, mq, mk, mv, mdy, stream);
    default: return launch_dq_t<128, 2, true>(a, tab, mq, mk, mv, mdy, stream);
  }
}

template cudaError_t launch_backward_dq<kSmallTable>(const BwdArgs&, const SeqTable<kSmallTable>&, const CUtensorMap&,
                                                     const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                     cudaStream_t);
template cudaError_t launch_backward_dq<kLargeTable>(const BwdArgs&, const SeqTable<kLargeTable>&, const CUtensorMap&,
                                                     const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                     cudaStream_t);

}  // namespace swa
