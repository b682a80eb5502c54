// swa_bwd_dkv.cu — sliding-window attention backward, key-major pass: dK, dV.
//
// Per (query tile i, key tile j) pair inside the BAND (PyPTO-Gym article,
// "反向公式"; aclnnFlashAttentionUnpaddingScoreGradV2 article §2.3), in the
// transposed orientation (one thread per key row):
//   S^T  = K Q^T                    P^T = exp2(S^T*scale*log2e - lse2)  (recomputed)
//   dP^T = V dY^T                   dS^T = P^T * (dP^T * z/keep - D)
//   dV  += (P * z/keep)^T dY        dK  += dS^T Q  (x scale at the end)
// lse2 = softmax_max*log2e + log2(softmax_sum) and D = rowsum(dY*O) come from
// the preprocess kernel.  dQ is computed by the query-major pass
// (swa_bwd_dq.cu), so nothing here accumulates through global memory.
//
// One CTA = one 128-row key tile of one (batch, head); it walks the query
// tiles of the band with dK / dV accumulating in TMEM.  Warps:
//   warps 0-7  compute: warp w owns TMEM lanes 32*(w%4).. (key rows) and query
//              columns 64*(w/4).. of each tile; then dV (w<4) or dK (w>=4)
//   warp  8    producer: K, V once; Q, dY by TMA through 2-stage rings, and
//              the tile's per-query lse2 / D (and dropout bits) into shared
//   warp  9    tcgen05 issuer
// TMEM: two 128-column regions R0, R1, dV [256,256+D), dK [256+D,256+2D).
// Tile i computes S^T into R(i%2) and dP^T into R((i+1)%2); once both are in
// registers, P^T and dS^T (bf16) are stored into R(i%2) and feed dV / dK as
// the TMEM A operand, while S^T(i+1) already runs in R((i+1)%2).
#include "swa_device.cuh"

namespace swa {
namespace {

template <int D>
struct DkvSmem {
  static constexpr int kTileBytes = kTileM * D * 2;
  alignas(1024) uint8_t k[kTileBytes];
  alignas(1024) uint8_t v[kTileBytes];
  alignas(1024) uint8_t q[2][kTileBytes];
  alignas(1024) uint8_t dy[2][kTileBytes];
  float lse2[2][kTileM];   // per query column of the tile in that stage (+inf: row outside)
  float dsum[2][kTileM];
  uint32_t keep[2][kTileM][4];  // dropout keep bits: [query row][key word]
  uint64_t kv_full, q_full[2], q_empty[2], dy_full[2], dy_empty[2], stat_full[2];
  uint64_t s_full, dp_full, sdp_loaded, pds_full, pds_free, mma_drain;
  uint32_t tmem_base;
};
static_assert(sizeof(DkvSmem<128>) + 1024 <= 232448, "shared memory budget");

constexpr int kThreads = 320;
constexpr int kComputeThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColDV = 256;
constexpr uint32_t kBarVote = 1;

__device__ __forceinline__ bool compute_wait(uint64_t* bar, uint32_t parity, int* err) {
  return named_barrier_and(kBarVote, kComputeThreads, mbar_wait(bar, parity, err, kErrBwdCompute));
}
__device__ __forceinline__ uint32_t region_s(int it) { return (it & 1) * 128u; }         // S^T, then P^T / dS^T
__device__ __forceinline__ uint32_t region_dp(int it) { return ((it + 1) & 1) * 128u; }  // dP^T

template <int D, bool DROP, int CAP>
__global__ void __launch_bounds__(kThreads, 1)
    swa_bwd_dkv_kernel(const BwdArgs a, const __grid_constant__ SeqTable<CAP> tab,
                       const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                       const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdy) {
  extern __shared__ uint8_t smem_raw[];
  DkvSmem<D>& s = *reinterpret_cast<DkvSmem<D>*>(align1024(smem_raw));
  constexpr int kTileBytes = DkvSmem<D>::kTileBytes;
  constexpr uint32_t kColDK = kColDV + D;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Geometry& g = a.g;
  const Item w = resolve_item(tab, a.g, static_cast<int>(blockIdx.x));
  const SeqInfo sq = w.s;
  const int j0 = w.tile * kTileN;
  const int j_last = min(j0 + kTileN - 1, sq.kv_len - 1);

  // query tiles that see this key tile
  int lo = 0, hi = sq.q_len - 1;
  if (g.sparse_mode == 4) {
    lo = max(lo, j0 - g.next);
    hi = min(hi, j_last + g.pre);
  }
  int q_t0 = 0, n_q = 0;
  if (lo <= hi) {
    q_t0 = lo / kTileM;
    n_q = hi / kTileM - q_t0 + 1;
  }

  if (threadIdx.x == 0) {
    mbar_init(&s.kv_full, 1);
    for (int st = 0; st < 2; ++st) {
      mbar_init(&s.q_full[st], 1);
      mbar_init(&s.q_empty[st], 1);
      mbar_init(&s.dy_full[st], 1);
      mbar_init(&s.dy_empty[st], 1);
      mbar_init(&s.stat_full[st], 32);
    }
    mbar_init(&s.s_full, 1);
    mbar_init(&s.dp_full, 1);
    mbar_init(&s.sdp_loaded, kComputeThreads);
    mbar_init(&s.pds_full, kComputeThreads);
    mbar_init(&s.pds_free, 1);
    mbar_init(&s.mma_drain, 1);
    fence_mbar_init();
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
    // -------------------------------------------------- producer (warp) --
    if (n_q > 0) {
      if (lane == 0) {
        tma_prefetch_desc(&mq);
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mv);
        tma_prefetch_desc(&mdy);
        mbar_arrive_expect_tx(&s.kv_full, 2 * kTileBytes);
        tma_rows<D>(s.k, &mk, &s.kv_full, g, w.b, w.n, sq.kv_start, j0);
        tma_rows<D>(s.v, &mv, &s.kv_full, g, w.b, w.n, sq.kv_start, j0);
      }
      int q_issued = 0, dy_issued = 0;
      for (int it = 0; it < n_q; ++it) {
        const int i0 = (q_t0 + it) * kTileM;
        const int st = it & 1;
        if (it >= 2 && !__all_sync(0xFFFFFFFFu, mbar_wait(&s.q_empty[st], ((it >> 1) - 1) & 1, a.err, kErrBwdLoad)))
          break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&s.q_full[st], kTileBytes);
          tma_rows<D>(s.q[st], &mq, &s.q_full[st], g, w.b, w.n, sq.q_start, i0);
        }
        ++q_issued;
        // per-query statistics (and keep bits) of this tile: 4 rows per lane
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int c = lane * 4 + k4;
          const int i = i0 + c;
          float l2 = INFINITY, dd = 0.f;
          uint32_t bits[4] = {0u, 0u, 0u, 0u};
          if (i < sq.q_len) {
            const int64_t si = stat_index(g, sq, w.b, w.n, i);
            l2 = a.lse2[si];
            dd = a.dsum[si];
            if (DROP) load_keep_bits(a.mask, sq, w.n, i, j0, bits);
          }
          s.lse2[st][c] = l2;
          s.dsum[st][c] = dd;
          if (DROP) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) s.keep[st][c][q4] = bits[q4];
          }
        }
        mbar_arrive(&s.stat_full[st]);
        if (it >= 2 &&
            !__all_sync(0xFFFFFFFFu, mbar_wait(&s.dy_empty[st], ((it >> 1) - 1) & 1, a.err, kErrBwdLoad)))
          break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&s.dy_full[st], kTileBytes);
          tma_rows<D>(s.dy[st], &mdy, &s.dy_full[st], g, w.b, w.n, sq.q_start, i0);
        }
        ++dy_issued;
      }
      // every copy issued has landed before the CTA may exit
      if (lane == 0) {
        mbar_wait_drain(&s.kv_full, 0);
        for (int st = 0; st < 2; ++st) {
          const int uq = (q_issued - st + 1) / 2, ud = (dy_issued - st + 1) / 2;
          if (uq > 0) mbar_wait_drain(&s.q_full[st], (uq - 1) & 1);
          if (ud > 0) mbar_wait_drain(&s.dy_full[st], (ud - 1) & 1);
        }
      }
    }
  } else if (warp == 9) {
    // ----------------------------------------------------- tcgen05 issuer --
    if (lane == 0 && n_q > 0) {
      constexpr uint32_t kIdT = idesc_bf16_f32(kTileN, kTileM, false, false);  // S^T, dP^T
      constexpr uint32_t kIdKV = idesc_bf16_f32(kTileN, D, false, true);       // dV, dK (A = P^T / dS^T in TMEM)
      const uint32_t k_addr = smem_u32(s.k), v_addr = smem_u32(s.v);
      auto issue_st = [&](int it) {  // S^T = K Q^T into region_s(it)
        const uint32_t q_addr = smem_u32(s.q[it & 1]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
          umma_bf16_ss(tmem + region_s(it), sdesc_sw128(k_addr + off, 16, 1024), sdesc_sw128(q_addr + off, 16, 1024),
                       kIdT, kk > 0);
        }
        umma_commit(&s.s_full);
      };
      auto issue_dpt = [&](int it) {  // dP^T = V dY^T into region_dp(it)
        const uint32_t dy_addr = smem_u32(s.dy[it & 1]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
          umma_bf16_ss(tmem + region_dp(it), sdesc_sw128(v_addr + off, 16, 1024),
                       sdesc_sw128(dy_addr + off, 16, 1024), kIdT, kk > 0);
        }
        umma_commit(&s.dp_full);
      };
      bool ok = mbar_wait(&s.kv_full, 0, a.err, kErrBwdMma) && mbar_wait(&s.q_full[0], 0, a.err, kErrBwdMma) &&
                mbar_wait(&s.dy_full[0], 0, a.err, kErrBwdMma);
      if (ok) {
        tc_fence_after_sync();
        issue_st(0);
        issue_dpt(0);
      }
      for (int it = 0; ok && it < n_q; ++it) {
        const int st = it & 1;
        const uint32_t ph = it & 1;
        // region_dp(it) is free once S^T(it) / dP^T(it) are in registers
        if (!mbar_wait(&s.sdp_loaded, ph, a.err, kErrBwdMma)) break;
        if (it + 1 < n_q) {
          if (!mbar_wait(&s.q_full[(it + 1) & 1], ((it + 1) >> 1) & 1, a.err, kErrBwdMma)) break;
          tc_fence_after_sync();
          issue_st(it + 1);
        }
        if (!mbar_wait(&s.pds_full, ph, a.err, kErrBwdMma)) break;
        tc_fence_after_sync();
        const uint32_t dy_addr = smem_u32(s.dy[st]), q_addr = smem_u32(s.q[st]);
        const uint32_t ra = tmem + region_s(it);
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk)  // dV += P^T dY  (K dim = query rows)
          umma_bf16_ts(tmem + kColDV, ra + kk * 8, sdesc_sw128(dy_addr + kk * 2048, kAtomBytes, 1024), kIdKV,
                       (it > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&s.dy_empty[st]);
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk)  // dK += dS^T Q
          umma_bf16_ts(tmem + kColDK, ra + 64 + kk * 8, sdesc_sw128(q_addr + kk * 2048, kAtomBytes, 1024), kIdKV,
                       (it > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&s.q_empty[st]);
        umma_commit(&s.pds_free);
        if (it + 1 < n_q) {  // dP^T(i+1) reuses region_s(it) once dV / dK(it) have read it
          if (!mbar_wait(&s.pds_free, ph, a.err, kErrBwdMma)) break;
          if (!mbar_wait(&s.dy_full[(it + 1) & 1], ((it + 1) >> 1) & 1, a.err, kErrBwdMma)) break;
          tc_fence_after_sync();
          issue_dpt(it + 1);
        }
      }
      umma_commit(&s.mma_drain);
      mbar_wait_drain(&s.mma_drain, 0);
    }
  } else {
    // ------------------------------------------- compute warps (0..7) -----
    const int wq = warp & 3, h = warp >> 2;  // lane quarter, query-column half
    const int r = wq * 32 + lane;            // TMEM lane = key row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int cbase = h * 64;                // query columns [cbase, cbase + 64) of each tile
    const float c = g.scale_log2;
    const int j = j0 + r;
    // queries that see key j: i - pre <= j <= i + next  <=>  j - next <= i <= j + pre
    int qlo = 0, qhi = sq.q_len - 1;
    if (g.sparse_mode == 4) {
      qlo = max(qlo, j - g.next);
      qhi = min(qhi, j + g.pre);
    }
    if (j >= sq.kv_len) {
      qlo = 1;
      qhi = 0;
    }
    bool ok = true;
    for (int it = 0; it < n_q; ++it) {
      const int st = it & 1;
      const int i0 = (q_t0 + it) * kTileM;
      const bool full = tile_fully_visible(g, sq, i0, j0);
      if (!compute_wait(&s.s_full, it & 1, a.err)) { ok = false; break; }
      if (!compute_wait(&s.stat_full[st], (it >> 1) & 1, a.err)) { ok = false; break; }
      tc_fence_after_sync();
      // ---- S^T -> P^T (registers)
      float p[64];
      {
        uint32_t s0[32], s1[32];
        tmem_ld_32x32b_x32(tmem + lane_off + region_s(it) + cbase, s0);
        tmem_ld_32x32b_x32(tmem + lane_off + region_s(it) + cbase + 32, s1);
        tmem_ld_wait(s0);
        tmem_ld_wait(s1);
#pragma unroll
        for (int t4 = 0; t4 < 16; ++t4) {
          const float4 l4 = *reinterpret_cast<const float4*>(&s.lse2[st][cbase + t4 * 4]);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int t = t4 * 4 + u;
            const int i = i0 + cbase + t;
            const bool vis = full || (i >= qlo && i <= qhi);
            const float sv = __uint_as_float(t < 32 ? s0[t] : s1[t - 32]);
            p[t] = vis ? ex2_approx(sv * c - lv[u]) : 0.f;
          }
        }
      }
      // ---- dP^T -> dS^T; P^T*z/keep and dS^T packed bf16
      if (!compute_wait(&s.dp_full, it & 1, a.err)) { ok = false; break; }
      tc_fence_after_sync();
      uint32_t pk[32], dk[32];
      {
        uint32_t d0[32], d1[32];
        tmem_ld_32x32b_x32(tmem + lane_off + region_dp(it) + cbase, d0);
        tmem_ld_32x32b_x32(tmem + lane_off + region_dp(it) + cbase + 32, d1);
        tmem_ld_wait(d0);
        tmem_ld_wait(d1);
        tc_fence_before_sync();
        mbar_arrive(&s.sdp_loaded);
#pragma unroll
        for (int t4 = 0; t4 < 16; ++t4) {
          const float4 d4 = *reinterpret_cast<const float4*>(&s.dsum[st][cbase + t4 * 4]);
          const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
          float pv[4], dsv[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int t = t4 * 4 + u;
            float dp = __uint_as_float(t < 32 ? d0[t] : d1[t - 32]);
            float pt = p[t];
            if (DROP) {
              const bool keep = (s.keep[st][cbase + t][wq] >> lane) & 1u;  // bit (query, key r)
              pt = keep ? p[t] * g.inv_keep : 0.f;
              dp = keep ? dp * g.inv_keep : 0.f;
            }
            pv[u] = pt;
            dsv[u] = p[t] * (dp - dv4[u]);
          }
          pk[t4 * 2] = pack_bf16x2(pv[0], pv[1]);
          pk[t4 * 2 + 1] = pack_bf16x2(pv[2], pv[3]);
          dk[t4 * 2] = pack_bf16x2(dsv[0], dsv[1]);
          dk[t4 * 2 + 1] = pack_bf16x2(dsv[2], dsv[3]);
        }
      }
      // ---- P^T, dS^T -> TMEM region_s(it) (its S^T is consumed)
      tmem_st_32x32b_x32(tmem + lane_off + region_s(it) + h * 32, pk);
      tmem_st_32x32b_x32(tmem + lane_off + region_s(it) + 64 + h * 32, dk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&s.pds_full);
    }
    if (ok && n_q > 0) ok = compute_wait(&s.pds_free, (n_q - 1) & 1, a.err);  // every MMA done
    if (ok) {
      tc_fence_after_sync();
      // epilogue: thread r owns key row j0 + r; warps 0-3 write dV, 4-7 dK
      const bool kv_valid = j < sq.kv_len;
      const uint32_t col = h == 0 ? kColDV : kColDK;
      const float mul = h == 0 ? 1.f : g.scale;
      __nv_bfloat16* dst = (h == 0 ? a.dv : a.dk) + kv_elem(g, sq, w.b, w.n, j);
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        float o[32];
        if (n_q > 0) {
          uint32_t t32[32];
          tmem_ld_32x32b_x32(tmem + lane_off + col + ch * 32, t32);
          tmem_ld_wait(t32);
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = __uint_as_float(t32[t]) * mul;
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = 0.f;
        }
        if (kv_valid) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) reinterpret_cast<uint4*>(dst + ch * 32)[q4] = pack8(&o[q4 * 8]);
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

template <int D, bool DROP, int CAP>
cudaError_t launch_dkv_t(const BwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, const CUtensorMap& mdy, cudaStream_t stream) {
  const size_t smem = sizeof(DkvSmem<D>) + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(swa_bwd_dkv_kernel<D, DROP, CAP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  swa_bwd_dkv_kernel<D, DROP, CAP><<<tab.n_items, kThreads, smem, stream>>>(a, tab, mq, mk, mv, mdy);
  return cudaGetLastError();
}

}  // namespace

template <int CAP>
cudaError_t launch_backward_dkv(const BwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq,
                                const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdy,
                                cudaStream_t stream) {
  if (tab.n_items == 0) return cudaSuccess;
  const bool drop = a.g.has_mask != 0;
  if (a.g.D == 64) return drop ? launch_dkv_t<64, true>(a, tab, mq, mk, mv, mdy, stream)
                               : launch_dkv_t<64, false>(a, tab, mq, mk, mv, mdy, stream);
  return drop ? launch_dkv_t<128, true>(a, tab, mq, mk, mv, mdy, stream)
              : launch_dkv_t<128, false>(a, tab, mq, mk, mv, mdy, stream);
}

template cudaError_t launch_backward_dkv<kSmallTable>(const BwdArgs&, const SeqTable<kSmallTable>&,
                                                      const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                      const CUtensorMap&, cudaStream_t);
template cudaError_t launch_backward_dkv<kLargeTable>(const BwdArgs&, const SeqTable<kLargeTable>&,
                                                      const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                      const CUtensorMap&, cudaStream_t);

}  // namespace swa
