// swa_bwd_dkv.cu — sliding-window attention backward, key-major pass: dK, dV.
//
// Per (query tile i, key tile j) pair inside the BAND (PyPTO-Gym article,
// "反向公式"; aclnnFlashAttentionUnpaddingScoreGradV2 article §2.3), in the
// transposed orientation (one thread per key row):
//   S^T  = K Q^T                    P^T = exp2(S^T*scale*log2e - lse2)  (recomputed)
//   dP^T = V dY^T                   dS^T = P^T * (dP^T * z/keep - D)
//   dV  += (P * z/keep)^T dY        dK  += dS^T Q  (x scale at the end)
// With dropout the 1/keep factor leaves the per-element work: the tiles carry
// (P*z)^T and P^T * (z*dP^T - keep*D), and the epilogues multiply dV by 1/keep
// and dK by scale/keep.
// lse2 = softmax_max*log2e + log2(softmax_sum) and D = rowsum(dY*O) come from
// the preprocess kernel.  dQ is computed by the query-major pass
// (swa_bwd_dq.cu), so nothing here accumulates through global memory.
//
// One CTA = one 128-row key tile of one (batch, head); it walks the query
// tiles of the band with dK / dV accumulating in TMEM.  Warps:
//   warps 0-7  compute: warp w owns TMEM lanes 32*(w%4).. (key rows) and query
//              columns 64*(w/4).. of each tile; then dV (w<4) or dK (w>=4)
//   warp  8    producer: K, V once; Q (3-stage ring) and dY (2 stages) by TMA,
//              and each tile's per-query lse2 / D (and dropout bits) into shared
//   warp  9    tcgen05 issuer of S^T and dP^T (SS)
//   warp 10    tcgen05 issuer of dV and dK (TS)
// TMEM: R 128-column regions (R = 2 at D = 128, 3 at D <= 64), then dV and
// dK (DkvTmem).  Query tile i lives in region i % R: S^T(i) is computed there;
// once every thread has it in registers, dP^T(i) is computed over it; each
// thread then stores its P^T / dS^T (bf16) into the very columns it read, and
// dV / dK take them as the TMEM A operand.  Issue order per tile: dP^T(i),
// S^T(i+1) (into its region, once dK(i+1-R) has finished reading it), dV(i),
// dK(i): the tensor pipe
// always has the next GEMM queued while the compute warps work.  Two issuing
// threads keep it fed: its queue is shallow, so every barrier wait of a
// single issuer between GEMMs left it idle.
//
// Shared memory: the seven 128-row tiles take all but 3 KB of the 227 KB a
// CTA may have; the barriers and per-query statistics are placed around them
// (DkvPlan), so the kernel needs no particular alignment of its dynamic
// shared-memory base.
#include "swa_device.cuh"

namespace swa {
namespace {

constexpr int kThreads = 352;
constexpr int kComputeThreads = 256;
constexpr uint32_t kTmemCols = 512;

// TMEM plan: kRegions 128-column regions, each holding one query tile's S^T,
// then dP^T, then P^T / dS^T; dV and dK after them.  At D = 128 the two
// accumulators take 256 columns and two regions fit; at D <= 64 a third
// region fits, so S^T(i+1) waits for dK(i-2) to release its region instead
// of dK(i-1).
template <int D>
struct DkvTmem {
  static constexpr int kRegions = D <= 64 ? 3 : 2;
  static constexpr uint32_t kColDV = kRegions * 128u;
  static constexpr uint32_t kColDK = kColDV + D;
  static_assert(kColDK + D <= kTmemCols, "TMEM plan");
};
constexpr size_t kMaxSmem = 232448;

// mbarrier slots
enum : int {
  kBarKvFull = 0,
  kBarQFull = 1,       // [3]
  kBarQEmpty = 4,      // [3]
  kBarDyFull = 7,      // [2]
  kBarDyEmpty = 9,     // [2]
  kBarStatFull = 11,   // [2]
  kBarGenFull = 13,    // [2] generated keep bits of the tile in that stage written (compute threads)
  kBarSFull = 15,      // [3] per region: the two issuers hand off there, so no waiter is a phase behind
  kBarPtFull = 18,     // [3]
  kBarDsFull = 21,     // [3]
  kBarRegionFree = 24, // [3]
  kBarDsHalf = 27,     // [3] the first 32-query half of each thread's dS^T columns stored
  kBarSLoaded = 30,
  kBarDpFull,
  kBarMmaDone,
  kBarDrainSdp,
  kBarDrainKv,
  kBarNever,  // completed by nothing: the target of the stall test hook
  kNumBars
};

// Shared-memory plan.  The tiles (K, V, the Q ring, the dY ring) need
// 1024-byte alignment (128-byte swizzle atoms); the small items (barriers,
// per-query statistics, keep bits) go into the gap before the first aligned
// address where they fit and after the tiles otherwise, so the layout fits the
// request for every 16-byte-aligned base of dynamic shared memory.
template <int D, bool DROP>
struct DkvPlan {
  static constexpr int kTileBytes = kTileM * D * 2;
  // a third Q stage lets Q(i+2) load while tile i computes; it does not fit
  // next to the dropout bits at D = 128
  static constexpr int kQStages = (DROP && D == 128) ? 2 : 3;
  static constexpr int kTiles = 2 + kQStages + 2;
  static constexpr size_t kTileRegion = static_cast<size_t>(kTiles) * kTileBytes;
  static constexpr size_t kBarBytes = ((kNumBars * 8 + 4) + 15) / 16 * 16;  // barriers + TMEM address slot
  static constexpr size_t kStatBytes = 2 * kTileM * 4;                      // lse2 (or D) of both stages
  static constexpr size_t kKeepBytes = DROP ? 2 * kTileM * 4 * 4 : 0;       // keep words of both stages
  static constexpr int kItems = DROP ? 4 : 3;
  static constexpr size_t item(int i) {
    return i == 0 ? kBarBytes : (i < 3 ? kStatBytes : kKeepBytes);  // barriers, lse2, D, keep bits
  }
  static constexpr size_t kSmallBytes = kBarBytes + 2 * kStatBytes + kKeepBytes;
  static constexpr size_t kSmem =
      kTileRegion + kSmallBytes + 1024 < kMaxSmem ? kTileRegion + kSmallBytes + 1024 : kMaxSmem;
  // every 16-byte base offset modulo 1024 leaves room for the greedy placement
  static constexpr bool fits() {
    for (size_t x = 0; x < 1024; x += 16) {
      size_t front = (1024 - x) & 1023;
      if (kSmem < front + kTileRegion) return false;
      size_t tail = kSmem - front - kTileRegion;
      for (int i = 0; i < kItems; ++i) {
        if (item(i) <= front) front -= item(i);
        else if (item(i) <= tail) tail -= item(i);
        else return false;
      }
    }
    return true;
  }
};
static_assert(DkvPlan<128, false>::fits() && DkvPlan<128, true>::fits(), "shared memory budget");
static_assert(DkvPlan<64, false>::fits() && DkvPlan<64, true>::fits(), "shared memory budget");

// Addresses of the plan's items; stage s of a ring or of the per-tile
// arrays is found by arithmetic (no run-time indexed pointer arrays, which
// would live in local memory).
template <int D, bool DROP>
struct DkvSmem {
  using P = DkvPlan<D, DROP>;
  uint8_t* tiles;  // K, V, Q stages, dY stages
  uint64_t* bar;
  uint32_t* tmem_slot;
  float* lse2_base;    // [2][128]: per query column of the tile in that stage (+inf: row outside)
  float* dsum_base;    // [2][128]
  uint32_t* keep_base;  // [2][128][4]: dropout keep bits, [query row][key word]

  __device__ explicit DkvSmem(uint8_t* raw) {
    const uintptr_t base = reinterpret_cast<uintptr_t>(raw);
    tiles = reinterpret_cast<uint8_t*>((base + 1023) & ~uintptr_t(1023));
    uint8_t* front = raw;
    size_t front_left = static_cast<size_t>(tiles - raw);
    uint8_t* tail = tiles + P::kTileRegion;
    auto take = [&](size_t n) -> uint8_t* {  // the same greedy rule DkvPlan::fits checks
      uint8_t* p;
      if (n <= front_left) {
        p = front;
        front += n;
        front_left -= n;
      } else {
        p = tail;
        tail += n;
      }
      return p;
    };
    uint8_t* b = take(P::kBarBytes);
    bar = reinterpret_cast<uint64_t*>(b);
    tmem_slot = reinterpret_cast<uint32_t*>(b + kNumBars * 8);
    lse2_base = reinterpret_cast<float*>(take(P::kStatBytes));
    dsum_base = reinterpret_cast<float*>(take(P::kStatBytes));
    keep_base = DROP ? reinterpret_cast<uint32_t*>(take(P::kKeepBytes)) : nullptr;
  }
  __device__ uint8_t* k() const { return tiles; }
  __device__ uint8_t* v() const { return tiles + P::kTileBytes; }
  __device__ uint8_t* q(int st) const { return tiles + (2 + st) * P::kTileBytes; }
  __device__ uint8_t* dy(int st) const { return tiles + (2 + P::kQStages + st) * P::kTileBytes; }
  __device__ float* lse2(int st) const { return lse2_base + st * kTileM; }
  __device__ float* dsum(int st) const { return dsum_base + st * kTileM; }
  __device__ uint32_t* keep(int st) const { return keep_base + st * kTileM * 4; }
};

// Warp-uniform bounded wait of the compute warps.  A warp vote (not a
// CTA-wide barrier) keeps each warp converged for its warp-collective TMEM
// accesses; no compute step reads what another warp wrote in TMEM.
__device__ __forceinline__ bool compute_wait(uint64_t* bar, uint32_t parity, int* err) {
  return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, err, kErrBwdCompute));
}
// Region of step it, and the phase parity of its per-region barriers.
template <int R>
__device__ __forceinline__ int region_of(int it) { return it % R; }
template <int R>
__device__ __forceinline__ uint32_t region_phase(int it) { return static_cast<uint32_t>((it / R) & 1); }

template <int D, int DM, bool F16, int CAP>
__global__ void __launch_bounds__(kThreads, 1)
    swa_bwd_dkv_kernel(const BwdArgs a, const __grid_constant__ SeqTable<CAP> tab,
                       const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                       const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdy) {
  constexpr bool DROP = DM != 0;
  using Plan = DkvPlan<D, DROP>;
  constexpr int kQS = Plan::kQStages;
  constexpr int kTileBytes = Plan::kTileBytes;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const DkvSmem<D, DROP> s(smem_raw);
  uint64_t* const bar = s.bar;
  constexpr int kR = DkvTmem<D>::kRegions;
  constexpr uint32_t kColDV = DkvTmem<D>::kColDV, kColDK = DkvTmem<D>::kColDK;
  auto region = [](int it) { return static_cast<uint32_t>(region_of<kR>(it)) * 128u; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_launch_dependents();  // the query-major pass reads nothing this grid writes
  const Geometry& g = a.g;
  const Item w = resolve_item(tab, a.g, static_cast<int>(blockIdx.x), a.g.N_kv);  // w.n: key/value head
  const SeqInfo sq = w.s;
  const int j0 = w.tile * kTileN;

  // query tiles that see this key tile
  int q_t0, n_q;
  query_tiles_of_key_tile(g, sq, w.tile, &q_t0, &n_q);
  // The CTA walks those query tiles for each query head that reads this
  // key/value head (one head without grouping): step it is query tile
  // q_t0 + it % n_q of query head w.n * group + it / n_q, and dK / dV sum
  // over all of them in TMEM.
  const int n_it = g.group * n_q;

  // The producer's lane initialises the barriers and issues the loads of K,
  // V and the first Q and dY tiles before the CTA-wide barrier, so their
  // latency runs while TMEM is allocated.
  if (warp == 8 && lane == 0) {
    mbar_init(&bar[kBarKvFull], 1);
    for (int st = 0; st < kQS; ++st) {
      mbar_init(&bar[kBarQFull + (st)], 1);
      mbar_init(&bar[kBarQEmpty + (st)], 1);
    }
    for (int st = 0; st < 2; ++st) {
      mbar_init(&bar[kBarDyFull + (st)], 1);
      mbar_init(&bar[kBarDyEmpty + (st)], 1);
      mbar_init(&bar[kBarStatFull + (st)], 32);
      mbar_init(&bar[kBarGenFull + (st)], kComputeThreads);
    }
    mbar_init(&bar[kBarSLoaded], kComputeThreads);
    mbar_init(&bar[kBarDpFull], 1);
    for (int r = 0; r < kR; ++r) {
      mbar_init(&bar[kBarSFull + (r)], 1);
      mbar_init(&bar[kBarPtFull + (r)], kComputeThreads);
      mbar_init(&bar[kBarDsFull + (r)], kComputeThreads);
      mbar_init(&bar[kBarDsHalf + (r)], kComputeThreads);
      mbar_init(&bar[kBarRegionFree + (r)], 1);
    }
    mbar_init(&bar[kBarMmaDone], 1);
    mbar_init(&bar[kBarDrainSdp], 1);
    mbar_init(&bar[kBarDrainKv], 1);
    mbar_init(&bar[kBarNever], 1);
    fence_mbar_init();
    if (n_q > 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
      tma_prefetch_desc(&mdy);
      mbar_arrive_expect_tx(&bar[kBarKvFull], 2 * kTileBytes);
      tma_rows<D>(s.k(), &mk, &bar[kBarKvFull], g, w.b, w.n, sq.kv_start, j0);
      tma_rows<D>(s.v(), &mv, &bar[kBarKvFull], g, w.b, w.n, sq.kv_start, j0);
      const int i0 = q_t0 * kTileM, qn = w.n * g.group;  // step 0
      mbar_arrive_expect_tx(&bar[kBarQFull], kTileBytes);
      tma_rows<D>(s.q(0), &mq, &bar[kBarQFull], g, w.b, qn, sq.q_start, i0);
      mbar_arrive_expect_tx(&bar[kBarDyFull], kTileBytes);
      tma_rows<D>(s.dy(0), &mdy, &bar[kBarDyFull], g, w.b, qn, sq.q_start, i0);
    }
  }
  if (warp == 9) {
    tmem_alloc(s.tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *s.tmem_slot;

  if (warp == 8) {
    // -------------------------------------------------- producer (warp) --
    // the per-query statistics below come from the preprocess grid; every
    // lane waits for it (so this grid also completes only after it has)
    griddep_wait();
    if (n_q > 0) {
      int q_issued = 0, dy_issued = 0;
      for (int it = 0; it < n_it; ++it) {
        const int i0 = (q_t0 + it % n_q) * kTileM;
        const int qn = w.n * g.group + it / n_q;  // query head of this step
        const int qs = it % kQS;
        // Q(it) reuses the stage of Q(it - kQS), free once dK of that tile is done
        if (it >= kQS &&
            !__all_sync(0xFFFFFFFFu, mbar_wait(&bar[kBarQEmpty + (qs)], ((it / kQS) - 1) & 1, a.err, kErrBwdLoad)))
          break;
        if (lane == 0 && it > 0) {  // Q(0) went out before the CTA-wide barrier
          mbar_arrive_expect_tx(&bar[kBarQFull + (qs)], kTileBytes);
          tma_rows<D>(s.q(qs), &mq, &bar[kBarQFull + (qs)], g, w.b, qn, sq.q_start, i0);
        }
        ++q_issued;
        // dY reuses stage (it & 1) once dV(it - 2), its last reader, is done
        const int st = it & 1;
        if (it >= 2 &&
            !__all_sync(0xFFFFFFFFu, mbar_wait(&bar[kBarDyEmpty + (st)], ((it >> 1) - 1) & 1, a.err, kErrBwdLoad)))
          break;
        if (lane == 0 && it > 0) {  // so did dY(0)
          mbar_arrive_expect_tx(&bar[kBarDyFull + (st)], kTileBytes);
          tma_rows<D>(s.dy(st), &mdy, &bar[kBarDyFull + (st)], g, w.b, qn, sq.q_start, i0);
        }
        ++dy_issued;
        // per-query statistics (and keep bits) of this tile, 4 rows per lane:
        // loaded into registers first, then written into stage (it & 1) once
        // the compute warps have stored dS^T(it - 2).  That is their last read
        // of the stage (D is read while dS^T is formed, after dV(it - 2) may
        // already have finished), and the barrier cannot run a phase ahead:
        // its next phase needs a tile whose statistics are not written yet.
        float l2[4], dd[4];
        uint32_t bits[4][4];
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int i = i0 + lane * 4 + k4;
          l2[k4] = INFINITY;
          dd[k4] = 0.f;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) bits[k4][q4] = 0u;
          if (i < sq.q_len) {
            const int64_t si = ws_stat_index(g, sq, w.b, qn, i);
            if (in_bounds(si, 1, g.n_stats, a.err)) {
              l2[k4] = a.lse2[si];
              dd[k4] = a.dsum[si];
            }
            if constexpr (DROP) dd[k4] *= g.keep;  // the compute warps form P * (z dP - keep D)
            if constexpr (DM == 1) load_keep_bits(a.mask, sq, qn, i, j0, bits[k4], g.n_mask_bytes, a.err);
          }
        }
        if (it >= 2 && !__all_sync(0xFFFFFFFFu, mbar_wait(&bar[kBarDsFull + region_of<kR>(it - 2)],
                                                         region_phase<kR>(it - 2), a.err, kErrBwdLoad)))
          break;
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int c = lane * 4 + k4;
          s.lse2(st)[c] = l2[k4];
          s.dsum(st)[c] = dd[k4];
          if constexpr (DM == 1) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) s.keep(st)[(c) * 4 + (q4)] = bits[k4][q4];
          }
        }
        mbar_arrive(&bar[kBarStatFull + (st)]);
      }
      // every copy issued has landed before the CTA may exit
      if (lane == 0) {
        mbar_wait_drain(&bar[kBarKvFull], 0);
        for (int st = 0; st < kQS; ++st) {
          const int uq = (q_issued - st + kQS - 1) / kQS;
          if (uq > 0) mbar_wait_drain(&bar[kBarQFull + (st)], (uq - 1) & 1);
        }
        for (int st = 0; st < 2; ++st) {
          const int ud = (dy_issued - st + 1) / 2;
          if (ud > 0) mbar_wait_drain(&bar[kBarDyFull + (st)], (ud - 1) & 1);
        }
      }
    }
  } else if (warp == 9) {
    // ----------------------------------------------------- tcgen05 issuer --
    if (lane == 0 && n_q > 0) {
      constexpr uint32_t kIdT = idesc_f16_f32(kTileN, kTileM, false, false, F16);  // S^T, dP^T
      const uint32_t k_addr = smem_u32(s.k()), v_addr = smem_u32(s.v());
      const int nk = d_steps(g);
      auto issue_ss = [&](uint32_t d_col, uint32_t a_addr, uint32_t b_addr) {  // 128 x 128 x D, both K-major
        const uint64_t da = sdesc_sw128(a_addr, 16, 1024), db = sdesc_sw128(b_addr, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          if (kk >= nk) break;
          const uint32_t off = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
          umma_bf16_ss(tmem + d_col, sdesc_advance(da, off), sdesc_advance(db, off), kIdT, kk > 0);
        }
      };
      bool ok = mbar_wait(&bar[kBarKvFull], 0, a.err, kErrBwdMma) && mbar_wait(&bar[kBarQFull + (0)], 0, a.err, kErrBwdMma);
      if (ok) {
        tc_fence_after_sync();
        issue_ss(region(0), k_addr, smem_u32(s.q(0)));  // S^T(0) = K Q(0)^T
        umma_commit(&bar[kBarSFull + (0)]);
      }
      for (int it = 0; ok && it < n_it; ++it) {
        const int st = it & 1;
        // dP^T(it) over S^T(it), once every compute thread has read S^T(it)
        if (!mbar_wait(&bar[kBarSLoaded], it & 1, a.err, kErrBwdMma)) break;
        if (!mbar_wait(&bar[kBarDyFull + (st)], (it >> 1) & 1, a.err, kErrBwdMma)) break;
        tc_fence_after_sync();
        issue_ss(region(it), v_addr, smem_u32(s.dy(st)));  // dP^T = V dY^T
        umma_commit(&bar[kBarDpFull]);
        if (it + 1 < n_it) {
          // S^T(it+1) into its region, once dK(it+1-kR) has read it
          if (it + 1 >= kR && !mbar_wait(&bar[kBarRegionFree + region_of<kR>(it + 1 - kR)],
                                         region_phase<kR>(it + 1 - kR), a.err, kErrBwdMma))
            break;
          const int nq = (it + 1) % kQS;
          if (!mbar_wait(&bar[kBarQFull + (nq)], ((it + 1) / kQS) & 1, a.err, kErrBwdMma)) break;
          tc_fence_after_sync();
          issue_ss(region(it + 1), k_addr, smem_u32(s.q(nq)));
          umma_commit(&bar[kBarSFull + region_of<kR>(it + 1)]);
        }
      }
      umma_commit(&bar[kBarDrainSdp]);
      mbar_wait_drain(&bar[kBarDrainSdp], 0);
    }
  } else if (warp == 10) {
    // ------------------------------------------------- dV / dK issuer --
    if (lane == 0 && n_q > 0) {
      constexpr uint32_t kIdKV = idesc_f16_f32(kTileN, D, false, true, F16);  // A = P^T / dS^T in TMEM
      for (int it = 0; it < n_it; ++it) {
        const int st = it & 1, qs = it % kQS;
        // dV, dK from the P^T / dS^T the compute warps stored in region(it):
        // query columns [64h, 64h+64) of the tile hold P^T in columns
        // [64h, 64h+32) and dS^T in [64h+32, 64h+64), two bf16 per column.
        // P^T is stored first, so dV(it) runs while dS^T is computed.
        if (!mbar_wait(&bar[kBarPtFull + region_of<kR>(it)], region_phase<kR>(it), a.err, kErrBwdMma)) break;
        tc_fence_after_sync();
        const uint32_t ra = tmem + region(it);
        const uint64_t d_dy = sdesc_sw128(smem_u32(s.dy(st)), kAtomBytes, 1024);
        const uint64_t d_q = sdesc_sw128(smem_u32(s.q(qs)), kAtomBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk)  // dV += P^T dY  (K dim = query rows)
          umma_bf16_ts(tmem + kColDV, ra + (kk >> 2) * 64 + (kk & 3) * 8,
                       sdesc_advance(d_dy, kk * 2048), kIdKV, (it > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bar[kBarDyEmpty + (st)]);  // dP^T(it) read dY(it) too; it finished before P^T(it) existed
        // dK += dS^T Q in two parts: k-steps 0, 1, 4, 5 read the first
        // 32-query half of each warp's 64 dS^T columns, stored before the
        // second (DsHalf); k-steps 2, 3, 6, 7 the second (DsFull)
        auto dk_steps = [&](int k0) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int kk = k0 + (e & 1) + (e >> 1) * 4;
            umma_bf16_ts(tmem + kColDK, ra + (kk >> 2) * 64 + 32 + (kk & 3) * 8, sdesc_advance(d_q, kk * 2048),
                         kIdKV, (it > 0 || kk > 0) ? 1u : 0u);
          }
        };
        if (!mbar_wait(&bar[kBarDsHalf + region_of<kR>(it)], region_phase<kR>(it), a.err, kErrBwdMma)) break;
        tc_fence_after_sync();
        dk_steps(0);
        if (!mbar_wait(&bar[kBarDsFull + region_of<kR>(it)], region_phase<kR>(it), a.err, kErrBwdMma)) break;
        tc_fence_after_sync();
        dk_steps(2);
        umma_commit(&bar[kBarQEmpty + (qs)]);  // likewise S^T(it) for Q(it)
        umma_commit(&bar[kBarRegionFree + region_of<kR>(it)]);
        if (it == n_it - 1) umma_commit(&bar[kBarMmaDone]);
      }
      umma_commit(&bar[kBarDrainKv]);
      mbar_wait_drain(&bar[kBarDrainKv], 0);
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
    // Generated keep bits (DM == 2): thread (r, h) writes the words for keys
    // [64h, 64h + 64) of query row r of a tile into the stage the consumers
    // read (row r's four words, as the producer fills them from a mask).
    auto gen_tile_bits = [&](int it2) {
      const int stage = it2 & 1;
      const int qn = w.n * g.group + it2 / n_q;
      const int row_i = (q_t0 + it2 % n_q) * kTileM + r;
      uint32_t words[2];
      gen_keep_words<2>(g, stat_index(g, sq, w.b, qn, row_i), (j0 + cbase) >> 4, words);
      if constexpr (DROP) {
        s.keep(stage)[(r) * 4 + (2 * h)] = words[0];
        s.keep(stage)[(r) * 4 + (2 * h + 1)] = words[1];
      }
      mbar_arrive(&bar[kBarGenFull + (stage)]);
    };
    // test hook: wait on a barrier that nothing completes, so the bounded
    // wait runs out and the launch reports it
    if (g.stall & kStallKeyMajor) ok = compute_wait(&bar[kBarNever], 0, a.err);
    if (DM == 2 && n_it > 0) gen_tile_bits(0);
    for (int it = 0; ok && it < n_it; ++it) {
      const int st = it & 1;
      const int i0 = (q_t0 + it % n_q) * kTileM;
      const bool full = tile_fully_visible(g, sq, i0, j0);
      const uint32_t col = tmem + lane_off + region(it) + cbase;
      if (!compute_wait(&bar[kBarSFull + region_of<kR>(it)], region_phase<kR>(it), a.err)) { ok = false; break; }
      if (!compute_wait(&bar[kBarStatFull + (st)], (it >> 1) & 1, a.err)) { ok = false; break; }
      tc_fence_after_sync();
      // ---- S^T -> P^T (registers)
      float p[64];
      {
        uint32_t s0[32], s1[32];
        tmem_ld_32x32b_x32(col, s0);
        tmem_ld_32x32b_x32(col + 32, s1);
        tmem_ld_wait(s0);
        tmem_ld_wait(s1);
        tc_fence_before_sync();
        mbar_arrive(&bar[kBarSLoaded]);  // region(it) may now receive dP^T(it)
        // Two copies of the loop: tiles entirely inside the window (nearly
        // all of them) need no per-element mask.  In the masked copy the
        // exp2 is unconditional and the comparisons use non-short-circuit
        // operators, so the mask compiles to selects, not branches.
        if (full) {
#pragma unroll
          for (int t4 = 0; t4 < 16; ++t4) {
            const float4 l4 = *reinterpret_cast<const float4*>(&s.lse2(st)[cbase + t4 * 4]);
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int u = 0; u < 4; u += 2) {  // packed pairs: (s*c - lse2) in one f32x2 FMA
              const int t = t4 * 4 + u;
              float x0, x1;
              ffma2_bv(x0, x1, __uint_as_float(t < 32 ? s0[t] : s1[t - 32]),
                       __uint_as_float(t + 1 < 32 ? s0[t + 1] : s1[t - 31]), c, -lv[u], -lv[u + 1]);
              p[t] = ex2_approx(x0);
              p[t + 1] = ex2_approx(x1);
            }
          }
        } else {
          const int lo_t = qlo - (i0 + cbase), hi_t = qhi - (i0 + cbase);  // visible t in [lo_t, hi_t]
#pragma unroll
          for (int t4 = 0; t4 < 16; ++t4) {
            const float4 l4 = *reinterpret_cast<const float4*>(&s.lse2(st)[cbase + t4 * 4]);
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int t = t4 * 4 + u;
              const float e = ex2_approx(__uint_as_float(t < 32 ? s0[t] : s1[t - 32]) * c - lv[u]);
              p[t] = ((t >= lo_t) & (t <= hi_t)) ? e : 0.f;
            }
          }
        }
      }
      // ---- next tile's generated keep bits, into the stage tile it-1 used
      // once every thread is through with tile it-1 (its ds_full)
      if (DM == 2 && it + 1 < n_it) {
        if (it >= 1 &&
            !compute_wait(&bar[kBarDsFull + region_of<kR>(it - 1)], region_phase<kR>(it - 1), a.err)) {
          ok = false;
          break;
        }
        gen_tile_bits(it + 1);
      }
      // ---- dP^T -> dS^T; P^T*z/keep and dS^T packed bf16 into the same columns
      if (DM == 2 && !compute_wait(&bar[kBarGenFull + (st)], (it >> 1) & 1, a.err)) { ok = false; break; }
      if (!compute_wait(&bar[kBarDpFull], it & 1, a.err)) { ok = false; break; }
      tc_fence_after_sync();
      {
        // this thread's keep bits of the tile: bit t = (query cbase + t, key r).
        // The stage holds them query-major (word wq of query c: keys
        // 32 wq .. 32 wq + 31); lane l fetches query cbase + l's word and a
        // warp transpose hands lane k the bits of key 32 wq + k.
        uint32_t km[2] = {~0u, ~0u};
        if constexpr (DROP) {
          km[0] = warp_transpose_bits(s.keep(st)[(cbase + lane) * 4 + wq], lane);
          km[1] = warp_transpose_bits(s.keep(st)[(cbase + 32 + lane) * 4 + wq], lane);
        }
        // dS^T = P^T * (dP^T * z / keep - D) for the 32 query columns of one
        // half.  With dropout the loop forms P^T * (z dP^T - keep D), 1/keep
        // times dS^T, and the dK epilogue takes the 1/keep (the staged D
        // already holds keep D).
        auto ds_half = [&](int half, const uint32_t (&d)[32], uint32_t* dk) {
#pragma unroll
          for (int t4 = 0; t4 < 8; ++t4) {
            const int tb = half * 32 + t4 * 4;
            const float4 d4 = *reinterpret_cast<const float4*>(&s.dsum(st)[cbase + tb]);
            const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
            float dp[4], dsv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int t = tb + u;
              dp[u] = __uint_as_float(d[t4 * 4 + u]);
              if constexpr (DROP) dp[u] = keep_or_zero(dp[u], km[t >> 5], t & 31);
            }
#pragma unroll
            for (int u = 0; u < 4; u += 2)  // packed pairs
              fmulsub2(dsv[u], dsv[u + 1], p[tb + u], p[tb + u + 1], dp[u], dp[u + 1], dv4[u], dv4[u + 1]);
            dk[t4 * 2] = pack2<F16>(dsv[0], dsv[1]);
            dk[t4 * 2 + 1] = pack2<F16>(dsv[2], dsv[3]);
          }
        };
        uint32_t dk[32];
        {
          uint32_t d[32];  // dP^T columns [cbase, cbase + 32): read before P^T goes over them
          tmem_ld_32x32b_x32(col, d);
          tmem_ld_wait(d);
          // P^T * z first, so dV can start (the dV epilogue takes the 1/keep)
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t pk[16];
#pragma unroll
            for (int t2 = 0; t2 < 16; ++t2) {
              const int t = half * 32 + 2 * t2;
              float p0 = p[t], p1 = p[t + 1];
              if constexpr (DROP) {
                p0 = keep_or_zero(p0, km[t >> 5], t & 31);
                p1 = keep_or_zero(p1, km[(t + 1) >> 5], (t + 1) & 31);
              }
              pk[t2] = pack2<F16>(p0, p1);
            }
            tmem_st_32x32b_x16(col + half * 16, pk);
          }
          tmem_st_wait();
          tc_fence_before_sync();
          mbar_arrive(&bar[kBarPtFull + region_of<kR>(it)]);
          ds_half(0, d, dk);
        }
        {
          uint32_t d[32];  // dP^T columns [cbase + 32, cbase + 64), where dS^T goes
          tmem_ld_32x32b_x32(col + 32, d);
          tmem_ld_wait(d);
          // dP^T is in registers: the first half of dS^T goes out now, so dK
          // can start on it while the second half is formed
          tmem_st_32x32b_x16(col + 32, dk);
          tmem_st_wait();
          tc_fence_before_sync();
          mbar_arrive(&bar[kBarDsHalf + region_of<kR>(it)]);
          ds_half(1, d, dk + 16);
        }
        tmem_st_32x32b_x16(col + 48, dk + 16);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&bar[kBarDsFull + region_of<kR>(it)]);
    }
    if (ok && n_q > 0) ok = compute_wait(&bar[kBarMmaDone], 0, a.err);  // every MMA done
    // The eight compute warps agree on whether to write the epilogue: its
    // staging barrier below must see all eight or none.
    ok = named_barrier_and(1, kComputeThreads, ok);
    if (ok) {
      tc_fence_after_sync();
      // epilogue: thread r owns key row j0 + r; warps 0-3 write dV, 4-7 dK
      const bool kv_valid = j < sq.kv_len;
      const uint32_t dcol = h == 0 ? kColDV : kColDK;
      // the 1/keep of dropout left out of P^T z and dS^T (exactly 1 without dropout)
      const float mul = h == 0 ? g.inv_keep : g.scale * g.inv_keep;
      void* dbase = h == 0 ? a.dv : a.dk;
      // dV is staged in the V buffer and dK in the K buffer (every MMA is done)
      uint8_t* stage = h == 0 ? s.v() : s.k();
      const int64_t dst = kv_elem(g, sq, w.b, w.n, j);
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        if (ch * 32 >= g.D) break;  // columns past D are padding
        float o[32];
        if (n_q > 0) {
          uint32_t t32[32];
          tmem_ld_32x32b_x32(tmem + lane_off + dcol + ch * 32, t32);
          tmem_ld_wait(t32);
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = __uint_as_float(t32[t]) * mul;
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = 0.f;
        }
        if (g.out_f32) {
          if (kv_valid) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              if (ch * 32 + q4 * 8 < g.D && in_bounds(dst + ch * 32 + q4 * 8, 8, g.n_kv_elems, a.err))
                store8<F16>(dbase, dst + ch * 32 + q4 * 8, &o[q4 * 8], true);
          }
        } else {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            if (ch * 32 + q4 * 8 < g.D) st_chunk_sw128(stage, r, ch * 4 + q4, pack8<F16>(&o[q4 * 8]));
        }
      }
      if (!g.out_f32) {
        // each warp store writes whole rows (one row per thread would touch
        // 32 rows, 32 cache lines, per store); warps 0-3 store dV, 4-7 dK
        named_barrier_sync(1, kComputeThreads);
        constexpr int kChunks = D / 8;
        constexpr int kRowsPerStore = 32 / kChunks;
        const int c = lane % kChunks;
        for (int rr = wq * kRowsPerStore + lane / kChunks; rr < kTileN; rr += 4 * kRowsPerStore) {
          const int gj = j0 + rr;
          if (gj < sq.kv_len && c * 8 < g.D && in_bounds(kv_elem(g, sq, w.b, w.n, gj) + c * 8, 8, g.n_kv_elems, a.err))
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(dbase) + kv_elem(g, sq, w.b, w.n, gj) + c * 8) =
                ld_chunk_sw128(stage, rr, c);
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
cudaError_t launch_dkv_t(const BwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, const CUtensorMap& mdy, cudaStream_t stream) {
  constexpr size_t smem = DkvPlan<D, DM != 0>::kSmem;
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t e = set_smem_limit(swa_bwd_dkv_kernel<D, DM, F16, CAP>, smem, smem_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(swa_bwd_dkv_kernel<D, DM, F16, CAP>, dim3(tab.n_items), dim3(kThreads), smem, stream, a, tab, mq,
                    mk, mv, mdy);
}

}  // namespace

template <int CAP>
cudaError_t launch_backward_dkv(const BwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq,
                                const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdy,
                                cudaStream_t stream) {
  if (tab.n_items == 0) return cudaSuccess;
  // (drop mode, D, element type) -> one of the twelve instantiations
  switch ((drop_mode_of(a.g.has_mask, a.g.drop_gen) * 2 + (a.g.D <= 64 ? 0 : 1)) * 2 + (a.g.f16 ? 1 : 0)) {
    case 0: return launch_dkv_t<64, 0, false>(a, tab, mq, mk, mv, mdy, stream);
    case 1: return launch_dkv_t<64, 0, true>(a, tab, mq, mk, mv, mdy, stream);
    case 2: return launch_dkv_t<128, 0, false>(a, tab, mq, mk, mv, mdy, stream);
    case 3: return launch_dkv_t<128, 0, true>(a, tab, mq, mk, mv, mdy, stream);
    case 4: return launch_dkv_t<64, 1, false>(a, tab, mq, mk, mv, mdy, stream);
    case 5: return launch_dkv_t<64, 1, true>(a, tab, mq, mk, mv, mdy, stream);
    case 6: return launch_dkv_t<128, 1, false>(a, tab, mq, mk, mv, mdy, stream);
    case 7: return launch_dkv_t<128, 1, true>(a, tab, mq, mk, mv, mdy, stream);
    case 8: return launch_dkv_t<64, 2, false>(a, tab, mq, mk, mv, mdy, stream);
    case 9: return launch_dkv_t<64, 2, true>(a, tab, mq, mk, mv, mdy, stream);
    case 10: return launch_dkv_t<128, 2, false>(a, tab, mq, mk, mv, mdy, stream);
    default: return launch_dkv_t<128, 2, true>(a, tab, mq, mk, mv, mdy, stream);
  }
}

template cudaError_t launch_backward_dkv<kSmallTable>(const BwdArgs&, const SeqTable<kSmallTable>&,
                                                      const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                      const CUtensorMap&, cudaStream_t);
template cudaError_t launch_backward_dkv<kLargeTable>(const BwdArgs&, const SeqTable<kLargeTable>&,
                                                      const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                      const CUtensorMap&, cudaStream_t);

}  // namespace swa
