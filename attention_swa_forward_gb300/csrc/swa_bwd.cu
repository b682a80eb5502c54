// swa_bwd.cu — sliding-window attention backward on sm_103a.
//
// Per (query tile i, key tile j) pair inside the BAND (PyPTO-Gym article,
// "反向公式"; aclnnFlashAttentionUnpaddingScoreGradV2 article §2.3):
//   S  = Q K^T                      P  = exp2(S*scale*log2e - lse2)   (recomputed)
//   dP = dY V^T                     dS = P * (dP * z/keep - D)
//   dV += (P * z/keep)^T dY         dK += dS^T Q  (x scale at the end)
//   dQ += dS K                      (fp32 atomics; x scale in the convert pass)
// lse2 = softmax_max*log2e + log2(softmax_sum) and D = rowsum(dY*O) come from
// the preprocess kernel.
//
// One CTA = one 128-row key tile of one (batch, head) (key-major, so dK/dV
// stay in TMEM for the whole walk over the query tiles of the band).  Warps:
//   warps 0-3  P/dS computation (one thread per query row), dQ atomics, and
//              the dK/dV epilogue (one thread per key row)
//   warp  4    TMA producer: K, V once; Q and dY per query tile
//   warp  5    tcgen05 issuer
// TMEM columns: S [0,128), dP [128,256), dV [256,256+D), dK [256+D,256+2D),
// dQ [0,128) for D = 128 (S is consumed by then) or [384,448) for D = 64.
#include "swa_device.cuh"

namespace swa {
namespace {

template <int D>
struct BwdSmem {
  static constexpr int kTileBytes = kTileM * D * 2;
  alignas(1024) uint8_t k[kTileBytes];
  alignas(1024) uint8_t v[kTileBytes];
  alignas(1024) uint8_t q[kTileBytes];
  alignas(1024) uint8_t dy[kTileBytes];
  alignas(1024) uint8_t p[kTileM * kTileN * 2];   // P*z/keep, [query row][key], swizzled
  alignas(1024) uint8_t ds[kTileM * kTileN * 2];  // dS, same layout
  uint64_t kv_full, q_full, dy_full, q_empty, dy_empty, sdp_full, pds_full, dq_full, dq_read, mma_drain;
  uint32_t tmem_base;
};

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256;

template <int D, bool DROP, int CAP>
__global__ void __launch_bounds__(192, 1)
    swa_bwd_kernel(const BwdArgs a, const __grid_constant__ SeqTable<CAP> tab, const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdy) {
  extern __shared__ uint8_t smem_raw[];
  BwdSmem<D>& s = *reinterpret_cast<BwdSmem<D>*>(align1024(smem_raw));
  constexpr int kTileBytes = BwdSmem<D>::kTileBytes;
  constexpr uint32_t kColDK = kColDV + D;
  constexpr uint32_t kColDQ = (D == 128) ? 0u : 384u;
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
    mbar_init(&s.q_full, 1);
    mbar_init(&s.dy_full, 1);
    mbar_init(&s.q_empty, 1);
    mbar_init(&s.dy_empty, 1);
    mbar_init(&s.sdp_full, 1);
    mbar_init(&s.pds_full, kTileM);
    mbar_init(&s.dq_full, 1);
    mbar_init(&s.dq_read, kTileM);
    mbar_init(&s.mma_drain, 1);
    fence_mbar_init();
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
        if (it >= 1 && !mbar_wait(&s.q_empty, (it - 1) & 1, a.err, kErrBwdLoad)) break;
        mbar_arrive_expect_tx(&s.q_full, kTileBytes);
        tma_rows<D>(s.q, &mq, &s.q_full, g, w.b, w.n, sq.q_start, i0);
        ++q_issued;
        if (it >= 1 && !mbar_wait(&s.dy_empty, (it - 1) & 1, a.err, kErrBwdLoad)) break;
        mbar_arrive_expect_tx(&s.dy_full, kTileBytes);
        tma_rows<D>(s.dy, &mdy, &s.dy_full, g, w.b, w.n, sq.q_start, i0);
        ++dy_issued;
      }
      // every copy issued has landed before the CTA may exit
      mbar_wait_drain(&s.kv_full, 0);
      if (q_issued > 0) mbar_wait_drain(&s.q_full, (q_issued - 1) & 1);
      if (dy_issued > 0) mbar_wait_drain(&s.dy_full, (dy_issued - 1) & 1);
    }
  } else if (warp == 5) {
    // ----------------------------------------------------- tcgen05 issuer --
    if (lane == 0 && n_q > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(kTileM, kTileN, false, false);  // S, dP
      constexpr uint32_t kIdKV = idesc_bf16_f32(kTileN, D, true, true);        // dV, dK (A = P^T / dS^T)
      constexpr uint32_t kIdQ = idesc_bf16_f32(kTileM, D, false, true);        // dQ
      const uint32_t k_addr = smem_u32(s.k), v_addr = smem_u32(s.v), q_addr = smem_u32(s.q);
      const uint32_t dy_addr = smem_u32(s.dy), p_addr = smem_u32(s.p), ds_addr = smem_u32(s.ds);
      bool ok = mbar_wait(&s.kv_full, 0, a.err, kErrBwdMma);
      for (int it = 0; ok && it < n_q; ++it) {
        const uint32_t ph = it & 1;
        if (!mbar_wait(&s.q_full, ph, a.err, kErrBwdMma)) break;
        if (it >= 1 && !mbar_wait(&s.dq_read, (it - 1) & 1, a.err, kErrBwdMma)) break;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {  // S = Q K^T
          const uint32_t off = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
          umma_bf16_ss(tmem + kColS, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024), kIdS,
                       kk > 0);
        }
        if (!mbar_wait(&s.dy_full, ph, a.err, kErrBwdMma)) break;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {  // dP = dY V^T
          const uint32_t off = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
          umma_bf16_ss(tmem + kColDP, sdesc_sw128(dy_addr + off, 16, 1024), sdesc_sw128(v_addr + off, 16, 1024),
                       kIdS, kk > 0);
        }
        umma_commit(&s.sdp_full);
        if (!mbar_wait(&s.pds_full, ph, a.err, kErrBwdMma)) break;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk) {  // dV += P^T dY  (K dim = query rows)
          umma_bf16_ss(tmem + kColDV, sdesc_sw128(p_addr + kk * 2048, kAtomBytes, 1024),
                       sdesc_sw128(dy_addr + kk * 2048, kAtomBytes, 1024), kIdKV, (it > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&s.dy_empty);
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk) {  // dK += dS^T Q
          umma_bf16_ss(tmem + kColDK, sdesc_sw128(ds_addr + kk * 2048, kAtomBytes, 1024),
                       sdesc_sw128(q_addr + kk * 2048, kAtomBytes, 1024), kIdKV, (it > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {  // dQ = dS K  (K dim = keys)
          const uint32_t aoff = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
          umma_bf16_ss(tmem + kColDQ, sdesc_sw128(ds_addr + aoff, 16, 1024),
                       sdesc_sw128(k_addr + kk * 2048, kAtomBytes, 1024), kIdQ, kk > 0);
        }
        umma_commit(&s.q_empty);
        umma_commit(&s.dq_full);
      }
      umma_commit(&s.mma_drain);
      mbar_wait_drain(&s.mma_drain, 0);
    }
  } else {
    // ------------------------------------------------ P / dS, dQ, dK / dV --
    const int r = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float c = g.scale_log2;
    bool ok = true;
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
      if (!mbar_wait(&s.sdp_full, it & 1, a.err, kErrBwdCompute)) { ok = false; break; }
      tc_fence_after_sync();
#pragma unroll
      for (int ch = 0; ch < kTileN / 32; ++ch) {
        uint32_t sv[32], dpv[32];
        tmem_ld_32x32b_x32(tmem + lane_off + kColS + ch * 32, sv);
        tmem_ld_32x32b_x32(tmem + lane_off + kColDP + ch * 32, dpv);
        tmem_ld_wait(sv);
        tmem_ld_wait(dpv);
        float pt[32], dsv[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          const int jj = ch * 32 + t;
          const int j = j0 + jj;
          const bool vis = full || (j >= wlo && j <= whi);
          const float p = vis ? ex2_approx(__uint_as_float(sv[t]) * c - lse2) : 0.f;
          float dp = __uint_as_float(dpv[t]);
          float pk = p;
          if (DROP) {
            const bool keep = (bits[jj >> 5] >> (jj & 31)) & 1u;
            pk = keep ? p * g.inv_keep : 0.f;
            dp = keep ? dp * g.inv_keep : 0.f;
          }
          pt[t] = pk;
          dsv[t] = p * (dp - drow);
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          st_chunk_sw128(s.p, r, ch * 4 + q4, pack8(&pt[q4 * 8]));
          st_chunk_sw128(s.ds, r, ch * 4 + q4, pack8(&dsv[q4 * 8]));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(&s.pds_full);
      // dQ tile -> fp32 accumulator
      if (!mbar_wait(&s.dq_full, it & 1, a.err, kErrBwdCompute)) { ok = false; break; }
      tc_fence_after_sync();
      float* dqrow = a.dq_acc + q_elem(g, sq, w.b, w.n, i);
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t t32[32];
        tmem_ld_32x32b_x32(tmem + lane_off + kColDQ + ch * 32, t32);
        tmem_ld_wait(t32);
        if (row_valid) {
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            atomicAdd(reinterpret_cast<float4*>(dqrow + ch * 32 + q4 * 4),
                      make_float4(__uint_as_float(t32[q4 * 4 + 0]), __uint_as_float(t32[q4 * 4 + 1]),
                                  __uint_as_float(t32[q4 * 4 + 2]), __uint_as_float(t32[q4 * 4 + 3])));
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&s.dq_read);
    }
    if (ok) {
      // epilogue: thread r owns key row j0 + r (TMEM lane r of dK / dV)
      const int j = j0 + r;
      const bool kv_valid = j < sq.kv_len;
      const int64_t off = kv_elem(g, sq, w.b, w.n, j);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? kColDV : kColDK;
        const float mul = which == 0 ? 1.f : g.scale;
        __nv_bfloat16* dst = (which == 0 ? a.dv : a.dk) + off;
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
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool DROP, int CAP>
cudaError_t launch_bwd_t(const BwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, const CUtensorMap& mdy, cudaStream_t stream) {
  const size_t smem = sizeof(BwdSmem<D>) + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(swa_bwd_kernel<D, DROP, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  swa_bwd_kernel<D, DROP, CAP><<<tab.n_items, 192, smem, stream>>>(a, tab, mq, mk, mv, mdy);
  return cudaGetLastError();
}

}  // namespace

template <int CAP>
cudaError_t launch_backward(const BwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, const CUtensorMap& mdy, cudaStream_t stream) {
  if (tab.n_items == 0) return cudaSuccess;
  const bool drop = a.g.has_mask != 0;
  if (a.g.D == 64) return drop ? launch_bwd_t<64, true>(a, tab, mq, mk, mv, mdy, stream)
                               : launch_bwd_t<64, false>(a, tab, mq, mk, mv, mdy, stream);
  return drop ? launch_bwd_t<128, true>(a, tab, mq, mk, mv, mdy, stream)
              : launch_bwd_t<128, false>(a, tab, mq, mk, mv, mdy, stream);
}

template cudaError_t launch_backward<kSmallTable>(const BwdArgs&, const SeqTable<kSmallTable>&, const CUtensorMap&,
                                                  const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                  cudaStream_t);
template cudaError_t launch_backward<kLargeTable>(const BwdArgs&, const SeqTable<kLargeTable>&, const CUtensorMap&,
                                                  const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                  cudaStream_t);

}  // namespace swa
