// swa_bwd.cu — sliding-window attention backward on sm_103a.
//
// Per (query tile i, key tile j) pair inside the BAND (PyPTO-Gym article,
// "反向公式"; aclnnFlashAttentionUnpaddingScoreGradV2 article §2.3):
//   S  = Q K^T                      P  = exp2(S*scale*log2e - lse2)   (recomputed)
//   dP = dY V^T                     dS = P * (dP * z/keep - D)
//   dV += (P * z/keep)^T dY         dK += dS^T Q  (x scale at the end)
//   dQ += dS K                      (TMA reduce-add into fp32; x scale in the convert pass)
// lse2 = softmax_max*log2e + log2(softmax_sum) and D = rowsum(dY*O) come from
// the preprocess kernel.
//
// One CTA = one 128-row key tile of one (batch, head) (key-major, so dK/dV
// stay in TMEM for the whole walk over the query tiles of the band).  Warps:
//   warps 0-7  compute: warp w owns TMEM lanes 32*(w%4).. and key columns
//              64*(w/4).. of each tile (P, dS, dQ staging), then one of dV /
//              dK in the epilogue
//   warp  8    TMA producer: K, V once; Q (2 stages) and dY per query tile
//   warp  9    tcgen05 issuer
// S and dP share TMEM columns [0,128): S is read into registers, then dP is
// written over it.  dQ [128,128+D), dV [128+D,128+2D), dK [128+2D,128+3D).
//
// The issue order keeps the tensor core fed while the compute warps work:
//   dP(i) | S(i+1) (as soon as dP(i) is in registers) | dV(i) dK(i) dQ(i)
// and dQ(i-1) is drained (TMEM -> swizzled staging -> TMA reduce-add) while
// the tensor core works on tile i.  The staging area is the P / dS buffer,
// free between the end of a tile's MMAs and the next tile's P / dS writes.
#include <cstddef>

#include "swa_device.cuh"

namespace swa {
namespace {

template <int D>
struct BwdSmem {
  static constexpr int kTileBytes = kTileM * D * 2;
  static constexpr int kDyStages = (D == 128) ? 1 : 2;
  alignas(1024) uint8_t k[kTileBytes];
  alignas(1024) uint8_t v[kTileBytes];
  alignas(1024) uint8_t q[2][kTileBytes];
  alignas(1024) uint8_t dy[kDyStages][kTileBytes];
  alignas(1024) uint8_t p[kTileM * kTileN * 2];   // P*z/keep, [query row][key], swizzled
  alignas(1024) uint8_t ds[kTileM * kTileN * 2];  // dS, same layout (p and ds double as the dQ staging)
  uint64_t kv_full, q_full[2], q_empty[2], dy_full[2], dy_empty[2];
  uint64_t s_full, s_loaded, dp_full, dp_loaded, pds_full, dq_full, dq_free, mma_drain;
  uint32_t tmem_base;
};
static_assert(offsetof(BwdSmem<128>, ds) == offsetof(BwdSmem<128>, p) + kTileM * kTileN * 2,
              "dQ staging spans p and ds");
static_assert(sizeof(BwdSmem<128>) + 1024 <= 232448, "shared memory budget");

constexpr int kThreads = 320;
constexpr int kComputeThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColSP = 0, kColDQ = 128;
constexpr uint32_t kBarVote = 1, kBarStage = 2;  // named barriers of the compute warps

// Every wait of the compute warps goes through a vote so that all of them
// continue or all of them stop.
__device__ __forceinline__ bool compute_wait(uint64_t* bar, uint32_t parity, int* err) {
  return named_barrier_and(kBarVote, kComputeThreads, mbar_wait(bar, parity, err, kErrBwdCompute));
}

template <int D, bool DROP, int CAP>
__global__ void __launch_bounds__(kThreads, 1)
    swa_bwd_kernel(const BwdArgs a, const __grid_constant__ SeqTable<CAP> tab, const __grid_constant__ CUtensorMap mq,
                   const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                   const __grid_constant__ CUtensorMap mdy, const __grid_constant__ CUtensorMap mdq) {
  extern __shared__ uint8_t smem_raw[];
  BwdSmem<D>& s = *reinterpret_cast<BwdSmem<D>*>(align1024(smem_raw));
  constexpr int kTileBytes = BwdSmem<D>::kTileBytes;
  constexpr int kDyStages = BwdSmem<D>::kDyStages;
  constexpr uint32_t kColDV = kColDQ + D;
  constexpr uint32_t kColDK = kColDQ + 2 * D;
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
    }
    mbar_init(&s.s_full, 1);
    mbar_init(&s.s_loaded, kComputeThreads);
    mbar_init(&s.dp_full, 1);
    mbar_init(&s.dp_loaded, kComputeThreads);
    mbar_init(&s.pds_full, kComputeThreads);
    mbar_init(&s.dq_full, 1);
    mbar_init(&s.dq_free, kComputeThreads);
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
    // ------------------------------------------------------ TMA producer --
    if (lane == 0 && n_q > 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
      tma_prefetch_desc(&mdy);
      mbar_arrive_expect_tx(&s.kv_full, 2 * kTileBytes);
      tma_rows<D>(s.k, &mk, &s.kv_full, g, w.b, w.n, sq.kv_start, j0);
      tma_rows<D>(s.v, &mv, &s.kv_full, g, w.b, w.n, sq.kv_start, j0);
      int q_issued = 0, dy_issued = 0;
      for (int it = 0; it < n_q; ++it) {
        const int i0 = (q_t0 + it) * kTileM;
        const int qs = it & 1;
        if (it >= 2 && !mbar_wait(&s.q_empty[qs], ((it >> 1) - 1) & 1, a.err, kErrBwdLoad)) break;
        mbar_arrive_expect_tx(&s.q_full[qs], kTileBytes);
        tma_rows<D>(s.q[qs], &mq, &s.q_full[qs], g, w.b, w.n, sq.q_start, i0);
        ++q_issued;
        const int ds_ = it % kDyStages;
        if (it >= kDyStages &&
            !mbar_wait(&s.dy_empty[ds_], ((it / kDyStages) - 1) & 1, a.err, kErrBwdLoad))
          break;
        mbar_arrive_expect_tx(&s.dy_full[ds_], kTileBytes);
        tma_rows<D>(s.dy[ds_], &mdy, &s.dy_full[ds_], g, w.b, w.n, sq.q_start, i0);
        ++dy_issued;
      }
      // every copy issued has landed before the CTA may exit
      mbar_wait_drain(&s.kv_full, 0);
      for (int st = 0; st < 2; ++st) {
        const int uq = (q_issued - st + 1) / 2;
        if (uq > 0) mbar_wait_drain(&s.q_full[st], (uq - 1) & 1);
      }
      for (int st = 0; st < kDyStages; ++st) {
        const int ud = (dy_issued - st + kDyStages - 1) / kDyStages;
        if (ud > 0) mbar_wait_drain(&s.dy_full[st], (ud - 1) & 1);
      }
    }
  } else if (warp == 9) {
    // ----------------------------------------------------- tcgen05 issuer --
    if (lane == 0 && n_q > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(kTileM, kTileN, false, false);  // S, dP
      constexpr uint32_t kIdKV = idesc_bf16_f32(kTileN, D, true, true);        // dV, dK (A = P^T / dS^T)
      constexpr uint32_t kIdQ = idesc_bf16_f32(kTileM, D, false, true);        // dQ
      const uint32_t k_addr = smem_u32(s.k), v_addr = smem_u32(s.v);
      const uint32_t p_addr = smem_u32(s.p), ds_addr = smem_u32(s.ds);
      auto issue_s = [&](int qs) {  // S = Q K^T into the shared S / dP columns
        const uint32_t q_addr = smem_u32(s.q[qs]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
          umma_bf16_ss(tmem + kColSP, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024),
                       kIdS, kk > 0);
        }
        umma_commit(&s.s_full);
      };
      bool ok = mbar_wait(&s.kv_full, 0, a.err, kErrBwdMma) && mbar_wait(&s.q_full[0], 0, a.err, kErrBwdMma);
      if (ok) {
        tc_fence_after_sync();
        issue_s(0);
      }
      for (int it = 0; ok && it < n_q; ++it) {
        const int qs = it & 1, ds_ = it % kDyStages;
        const uint32_t ph = it & 1;
        if (!mbar_wait(&s.s_loaded, ph, a.err, kErrBwdMma)) break;
        if (!mbar_wait(&s.dy_full[ds_], (it / kDyStages) & 1, a.err, kErrBwdMma)) break;
        tc_fence_after_sync();
        const uint32_t dy_addr = smem_u32(s.dy[ds_]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {  // dP = dY V^T over the consumed S
          const uint32_t off = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
          umma_bf16_ss(tmem + kColSP, sdesc_sw128(dy_addr + off, 16, 1024), sdesc_sw128(v_addr + off, 16, 1024),
                       kIdS, kk > 0);
        }
        umma_commit(&s.dp_full);
        if (!mbar_wait(&s.dp_loaded, ph, a.err, kErrBwdMma)) break;
        if (it + 1 < n_q) {  // next tile's S while this tile's P / dS are computed
          if (!mbar_wait(&s.q_full[(it + 1) & 1], ((it + 1) >> 1) & 1, a.err, kErrBwdMma)) break;
          tc_fence_after_sync();
          issue_s((it + 1) & 1);
        }
        if (!mbar_wait(&s.pds_full, ph, a.err, kErrBwdMma)) break;
        tc_fence_after_sync();
        const uint32_t q_addr = smem_u32(s.q[qs]);
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk) {  // dV += P^T dY  (K dim = query rows)
          umma_bf16_ss(tmem + kColDV, sdesc_sw128(p_addr + kk * 2048, kAtomBytes, 1024),
                       sdesc_sw128(dy_addr + kk * 2048, kAtomBytes, 1024), kIdKV, (it > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&s.dy_empty[ds_]);
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk) {  // dK += dS^T Q
          umma_bf16_ss(tmem + kColDK, sdesc_sw128(ds_addr + kk * 2048, kAtomBytes, 1024),
                       sdesc_sw128(q_addr + kk * 2048, kAtomBytes, 1024), kIdKV, (it > 0 || kk > 0) ? 1u : 0u);
        }
        if (it >= 1 && !mbar_wait(&s.dq_free, (it - 1) & 1, a.err, kErrBwdMma)) break;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {  // dQ = dS K  (K dim = keys)
          const uint32_t aoff = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
          umma_bf16_ss(tmem + kColDQ, sdesc_sw128(ds_addr + aoff, 16, 1024),
                       sdesc_sw128(k_addr + kk * 2048, kAtomBytes, 1024), kIdQ, kk > 0);
        }
        umma_commit(&s.q_empty[qs]);
        umma_commit(&s.dq_full);
      }
      umma_commit(&s.mma_drain);
      mbar_wait_drain(&s.mma_drain, 0);
    }
  } else {
    // ------------------------------------------- compute warps (0..7) -----
    const int wq = warp & 3, h = warp >> 2;  // lane quarter, key-column half
    const int r = wq * 32 + lane;            // TMEM lane = row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int cbase = h * 64;                // key columns [cbase, cbase + 64) of each tile
    const float c = g.scale_log2;
    bool ok = true;

    // dQ of query tile t: TMEM -> swizzled fp32 staging -> TMA reduce-add.
    // Rows past the sequence hold exact zeros (P = dS = 0 there); rows past
    // the tensor are skipped by the copy engine.
    auto drain_dq = [&](int t) -> bool {
      if (!compute_wait(&s.dq_full, t & 1, a.err)) return false;
      tc_fence_after_sync();
      constexpr int kCols = D / 2;  // this warp's dQ columns
      uint32_t d0[32], d1[32];
      tmem_ld_32x32b_x32(tmem + lane_off + kColDQ + h * kCols, d0);
      if (kCols == 64) tmem_ld_32x32b_x32(tmem + lane_off + kColDQ + h * kCols + 32, d1);
      tmem_ld_wait(d0);
      if (kCols == 64) tmem_ld_wait(d1);
      tc_fence_before_sync();
      uint8_t* box = s.p + ((h * kCols) / 32) * kAtomBytes + r * 128;
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4)
        *reinterpret_cast<uint4*>(box + (((c4 ^ r) & 7) << 4)) =
            make_uint4(d0[c4 * 4 + 0], d0[c4 * 4 + 1], d0[c4 * 4 + 2], d0[c4 * 4 + 3]);
      if (kCols == 64) {
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          *reinterpret_cast<uint4*>(box + kAtomBytes + (((c4 ^ r) & 7) << 4)) =
              make_uint4(d1[c4 * 4 + 0], d1[c4 * 4 + 1], d1[c4 * 4 + 2], d1[c4 * 4 + 3]);
      }
      fence_proxy_async_smem();
      named_barrier_sync(kBarStage, kComputeThreads);
      if (threadIdx.x == 0) {
        tma_reduce_rows<D>(s.p, &mdq, g, w.b, w.n, sq.q_start, (q_t0 + t) * kTileM);
        bulk_commit_group();
        bulk_wait_read_all();
      }
      named_barrier_sync(kBarStage, kComputeThreads);  // staging may be overwritten now
      mbar_arrive(&s.dq_free);
      return true;
    };

    for (int it = 0; it < n_q; ++it) {
      const int i0 = (q_t0 + it) * kTileM;
      const int i = i0 + r;
      const bool row_valid = i < sq.q_len;
      int wlo, whi;
      key_window(g, sq, i, wlo, whi);
      float lse2 = INFINITY, drow = 0.f;
      uint32_t bits[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
      if (row_valid) {
        const int64_t si = stat_index(g, sq, w.b, w.n, i);
        lse2 = a.lse2[si];
        drow = a.dsum[si];
        if (DROP) load_keep_bits(a.mask, sq, w.n, i, j0, bits);
      }
      const bool full = tile_fully_visible(g, sq, i0, j0);

      // ---- S -> P (kept in registers)
      if (!compute_wait(&s.s_full, it & 1, a.err)) { ok = false; break; }
      tc_fence_after_sync();
      float p[64];
      {
        uint32_t s0[32], s1[32];
        tmem_ld_32x32b_x32(tmem + lane_off + kColSP + cbase, s0);
        tmem_ld_32x32b_x32(tmem + lane_off + kColSP + cbase + 32, s1);
        tmem_ld_wait(s0);
        tmem_ld_wait(s1);
        tc_fence_before_sync();
        mbar_arrive(&s.s_loaded);
#pragma unroll
        for (int t = 0; t < 64; ++t) {
          const int j = j0 + cbase + t;
          const bool vis = full || (j >= wlo && j <= whi);
          const float sv = __uint_as_float(t < 32 ? s0[t] : s1[t - 32]);
          p[t] = vis ? ex2_approx(sv * c - lse2) : 0.f;
        }
      }
      // ---- dQ of the previous tile, while this tile's dP is computed
      if (it >= 1 && !drain_dq(it - 1)) { ok = false; break; }

      // ---- dP -> dS; P and dS to shared memory
      if (!compute_wait(&s.dp_full, it & 1, a.err)) { ok = false; break; }
      tc_fence_after_sync();
      {
        uint32_t d0[32], d1[32];
        tmem_ld_32x32b_x32(tmem + lane_off + kColSP + cbase, d0);
        tmem_ld_32x32b_x32(tmem + lane_off + kColSP + cbase + 32, d1);
        tmem_ld_wait(d0);
        tmem_ld_wait(d1);
        tc_fence_before_sync();
        mbar_arrive(&s.dp_loaded);
        const uint32_t kb0 = h ? bits[2] : bits[0], kb1 = h ? bits[3] : bits[1];  // this half's keep bits
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          float pt[8], dsv[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int t = c8 * 8 + u;
            float dp = __uint_as_float(t < 32 ? d0[t] : d1[t - 32]);
            float pk = p[t];
            if (DROP) {
              const bool keep = ((t < 32 ? kb0 : kb1) >> (t & 31)) & 1u;
              pk = keep ? p[t] * g.inv_keep : 0.f;
              dp = keep ? dp * g.inv_keep : 0.f;
            }
            pt[u] = pk;
            dsv[u] = p[t] * (dp - drow);
          }
          st_chunk_sw128(s.p, r, h * 8 + c8, pack8(pt));
          st_chunk_sw128(s.ds, r, h * 8 + c8, pack8(dsv));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(&s.pds_full);
    }
    if (ok && n_q > 0) ok = drain_dq(n_q - 1);
    if (threadIdx.x == 0) bulk_wait_all();
    if (ok) {
      // epilogue: thread r owns key row j0 + r; warps 0-3 write dV, 4-7 dK
      const int j = j0 + r;
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
cudaError_t launch_bwd_t(const BwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, const CUtensorMap& mdy, const CUtensorMap& mdq, cudaStream_t stream) {
  const size_t smem = sizeof(BwdSmem<D>) + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(swa_bwd_kernel<D, DROP, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  swa_bwd_kernel<D, DROP, CAP><<<tab.n_items, kThreads, smem, stream>>>(a, tab, mq, mk, mv, mdy, mdq);
  return cudaGetLastError();
}

}  // namespace

template <int CAP>
cudaError_t launch_backward(const BwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, const CUtensorMap& mdy, const CUtensorMap& mdq,
                            cudaStream_t stream) {
  if (tab.n_items == 0) return cudaSuccess;
  const bool drop = a.g.has_mask != 0;
  if (a.g.D == 64) return drop ? launch_bwd_t<64, true>(a, tab, mq, mk, mv, mdy, mdq, stream)
                               : launch_bwd_t<64, false>(a, tab, mq, mk, mv, mdy, mdq, stream);
  return drop ? launch_bwd_t<128, true>(a, tab, mq, mk, mv, mdy, mdq, stream)
              : launch_bwd_t<128, false>(a, tab, mq, mk, mv, mdy, mdq, stream);
}

template cudaError_t launch_backward<kSmallTable>(const BwdArgs&, const SeqTable<kSmallTable>&, const CUtensorMap&,
                                                  const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                  const CUtensorMap&, cudaStream_t);
template cudaError_t launch_backward<kLargeTable>(const BwdArgs&, const SeqTable<kLargeTable>&, const CUtensorMap&,
                                                  const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                  const CUtensorMap&, cudaStream_t);

}  // namespace swa
