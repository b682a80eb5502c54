// swa_aux.cu — the memory-bound pass before the backward kernels.
//
//  * preprocess: per query row, D = rowsum(dY * O) (PyPTO-Gym article,
//    "反向公式") and lse2 = softmax_max*log2(e) + log2(softmax_sum) (+inf for
//    an empty row, so that the recomputed P is 0), stored head-major.
//
// Both layouts address a query row (b, n, i) / (t, n) the same way once
// flattened: row id r -> elements [r*D, r*D + D), statistics index r.
#include "swa_internal.h"
#include "swa_device.cuh"

namespace swa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Two packed elements (bf16 or fp16) to floats.
template <bool F16>
__device__ __forceinline__ float2 unpack2(uint32_t v) {
  if constexpr (F16) return __half22float2(*reinterpret_cast<const __half2*>(&v));
  else return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
}

// D = rowsum(dY * O) and lse2 per query row, by bulk copies.  One CTA of 4
// warps per chunk of prep_chunk_rows(DP) rows (DP = 64 or 128, the head dim
// rounded up to one of them): up to 16 KB of dY, 16 KB of O and the chunk's
// softmax_max / softmax_sum, fetched by one thread with cp.async.bulk into
// shared memory.  Six CTAs fit an SM (shared memory), so up to six chunks
// are in flight per SM without holding them in registers, and the CTAs stay
// short, so that the grid fills SMs freed by kernels of other streams as
// they come.  Warp w reduces rows [w*R/4, (w+1)*R/4) of the chunk (4
// elements per lane over DP/4 lanes, those past D idle, then a butterfly
// over the row's lanes), lane t ends up holding row t's D and writes D and
// lse2.  kExact: D == DP, known at compile time.
constexpr int kPrepThreads = 128;
__host__ __device__ constexpr int prep_chunk_rows(int D) { return 8192 / D; }
__host__ __device__ constexpr size_t prep_bulk_smem(int D) {
  return 2 * static_cast<size_t>(prep_chunk_rows(D)) * D * 2 + 2 * static_cast<size_t>(prep_chunk_rows(D)) * 4 + 16;
}
static_assert(prep_bulk_smem(64) <= 48 * 1024 && prep_bulk_smem(128) <= 48 * 1024, "default launch limit");

// Bounded wait of the preprocess.  It does not consult the error word, which
// block 0 of this grid clears at its start, possibly after this block began.
__device__ __forceinline__ bool prep_wait(uint64_t* bar, uint32_t parity, int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(err, 0, static_cast<int32_t>(kErrPrepLoad));
      return false;
    }
  return true;
}

template <int DP, bool F16, bool kExact>
__global__ void __launch_bounds__(kPrepThreads) swa_prep_bulk_kernel(const PrepArgs a) {
  constexpr int kRows = prep_chunk_rows(DP);         // 64 or 128
  constexpr uint32_t kTileBytes = kRows * DP * 2;    // 16 KB: the stage of each tensor
  constexpr int kLanesPerRow = DP / 4;               // 8 bytes of each tensor per lane
  constexpr int kRowsPerIter = 32 / kLanesPerRow;    // 1 or 2 rows per warp step
  constexpr int kRowsPerWarp = kRows / (kPrepThreads / 32);  // 16 or 32
  static_assert(kRowsPerWarp <= 32 && kRowsPerWarp % kRowsPerIter == 0, "chunk split");
  const int D = kExact ? DP : a.g.D;  // a multiple of 8, at most DP
  extern __shared__ __align__(128) uint8_t smem[];
  const uint8_t* sdy = smem;
  const uint8_t* so = smem + kTileBytes;
  const float* s_max = reinterpret_cast<const float*>(smem + 2 * kTileBytes);
  const float* s_sum = s_max + kRows;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + 2 * kTileBytes + 2 * kRows * 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kRows;
  const int nrows = static_cast<int>(a.rows - row0 < kRows ? a.rows - row0 : kRows);
  const int nstat = nrows & ~3;  // statistics of whole 4-row groups come by bulk copy (16-byte sizes)
  if (threadIdx.x == 0) {
    mbar_init(full, 1);
    fence_mbar_init();
  }
  __syncthreads();
  griddep_wait();  // dY, O and the statistics come from earlier grids
  griddep_launch_dependents();
  if (!SWA_CHECKS && blockIdx.x == 0 && threadIdx.x == 0) *a.err = 0;  // fresh error word for this backward call
  if (threadIdx.x == 0) {
    const uint32_t tile = static_cast<uint32_t>(nrows) * D * 2;
    const bool ok = in_bounds(row0 * D, static_cast<int64_t>(nrows) * D, a.g.n_q_elems, a.err) &&
                    in_bounds(row0, nstat, a.g.n_stats, a.err);
    mbar_arrive_expect_tx(full, ok ? 2 * tile + 2 * nstat * 4 : 0);
    if (ok) {  // (the bounds-checked build skips the chunk; its status reports it)
      bulk_load(smem, a.dy + row0 * D, tile, full);
      bulk_load(smem + kTileBytes, a.out + row0 * D, tile, full);
      if (nstat > 0) {
        bulk_load(smem + 2 * kTileBytes, a.smax + row0, nstat * 4, full);
        bulk_load(smem + 2 * kTileBytes + kRows * 4, a.ssum + row0, nstat * 4, full);
      }
    }
  }
  if (!prep_wait(full, 0, a.err)) {
    if (threadIdx.x == 0) mbar_wait_drain(full, 0);  // copies in flight land before the CTA exits
    return;
  }
  float d_mine = 0.f;  // lane t < kRowsPerWarp: D of the warp's row t
#pragma unroll
  for (int it = 0; it < kRowsPerWarp / kRowsPerIter; ++it) {
    const int r = warp * kRowsPerWarp + it * kRowsPerIter + lane / kLanesPerRow;
    const int c = (lane % kLanesPerRow) * 4;  // first of the lane's 4 elements
    const int off = (r * D + c) * 2;
    uint2 dv = make_uint2(0u, 0u), ov = make_uint2(0u, 0u);
    if (kExact || c < D) {
      dv = *reinterpret_cast<const uint2*>(sdy + off);
      ov = *reinterpret_cast<const uint2*>(so + off);
    }
    const float2 d0 = unpack2<F16>(dv.x), d1 = unpack2<F16>(dv.y);
    const float2 o0 = unpack2<F16>(ov.x), o1 = unpack2<F16>(ov.y);
    float acc = d0.x * o0.x;
    acc = fmaf(d0.y, o0.y, acc);
    acc = fmaf(d1.x, o1.x, acc);
    acc = fmaf(d1.y, o1.y, acc);
#pragma unroll
    for (int m = kLanesPerRow / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, m);
    if constexpr (kRowsPerIter == 1) {
      if (lane == it) d_mine = acc;
    } else {  // lanes 0-15 hold row 2*it, lanes 16-31 row 2*it + 1; lanes 2*it and 2*it + 1 take them
      const float other = __shfl_xor_sync(0xFFFFFFFFu, acc, 16);
      const float even = lane < 16 ? acc : other, odd = lane < 16 ? other : acc;
      if (lane == 2 * it) d_mine = even;
      if (lane == 2 * it + 1) d_mine = odd;
    }
  }
  const int rloc = warp * kRowsPerWarp + lane;
  if (lane < kRowsPerWarp && rloc < nrows) {
    const int64_t row = row0 + rloc;
    const int64_t ws = a.g.layout == 0 ? row : (row % a.g.N) * a.g.T_q + row / a.g.N;
    float m, l;
    if (rloc < nstat) {
      m = s_max[rloc];
      l = s_sum[rloc];
    } else {  // past the tensor's last whole 4-row group: plain loads
      const bool in = in_bounds(row, 1, a.g.n_stats, a.err);
      m = in ? a.smax[row] : 0.f;
      l = in ? a.ssum[row] : 0.f;
    }
    if (in_bounds(ws, 1, a.g.n_stats, a.err)) {
      a.dsum[ws] = d_mine;
      a.lse2[ws] = (l > 0.f) ? m * kLog2e + __log2f(l) : INFINITY;
    }
  }
}

// The keep mask a seed / offset pair stands for, in the packed drop_mask
// layout: thread = one query row of a 128-row tile; it generates its row's
// keep bits 16 keys at a time and ORs them into the zeroed 32-bit words (a
// 16-bit group may straddle two words).
template <int CAP>
__global__ void __launch_bounds__(128) swa_dropmask_kernel(const MaskGenArgs a, const __grid_constant__ SeqTable<CAP> tab) {
  const Geometry& g = a.g;
  const Item w = resolve_item(tab, g, static_cast<int>(blockIdx.x), g.N);
  const SeqInfo sq = w.s;
  const int i = w.tile * kTileM + static_cast<int>(threadIdx.x);
  if (i >= sq.q_len) return;
  const int64_t row = stat_index(g, sq, w.b, w.n, i);
  const int64_t e_row = sq.mask_base + (static_cast<int64_t>(w.n) * sq.q_len + i) * sq.kv_len;
  const int nblk = (sq.kv_len + 15) / 16;
  for (int kb = 0; kb < nblk; ++kb) {
    uint32_t bits = gen_keep16(g, row, kb);
    const int cnt = min(16, sq.kv_len - kb * 16);
    if (cnt < 16) bits &= (1u << cnt) - 1u;
    if (!bits) continue;
    const int64_t e = e_row + kb * 16;
    const int sh = static_cast<int>(e & 31);
    atomicOr(&a.mask[e >> 5], bits << sh);
    if (sh > 16) atomicOr(&a.mask[(e >> 5) + 1], bits >> (32 - sh));
  }
}

}  // namespace

template <int CAP>
cudaError_t launch_dropout_mask(const MaskGenArgs& a, const SeqTable<CAP>& tab, cudaStream_t stream) {
  if (tab.n_items == 0) return cudaSuccess;
  swa_dropmask_kernel<CAP><<<tab.n_items, 128, 0, stream>>>(a, tab);
  return cudaGetLastError();
}
template cudaError_t launch_dropout_mask<kSmallTable>(const MaskGenArgs&, const SeqTable<kSmallTable>&, cudaStream_t);
template cudaError_t launch_dropout_mask<kLargeTable>(const MaskGenArgs&, const SeqTable<kLargeTable>&, cudaStream_t);

// fp32 -> bf16, eight elements (two 16-byte loads, one 16-byte store) per
// thread and grid-stride step.
__global__ void __launch_bounds__(256) swa_to_bf16_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out,
                                                          int64_t n8) {
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n8;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(in) + 2 * k);
    const float4 b = __ldg(reinterpret_cast<const float4*>(in) + 2 * k + 1);
    const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    reinterpret_cast<uint4*>(out)[k] = pack8<false>(x);
  }
}

cudaError_t launch_to_bf16(const float* in, __nv_bfloat16* out, int64_t n, cudaStream_t stream) {
  const int64_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  const int64_t want = (n8 + 255) / 256;
  const unsigned grid = static_cast<unsigned>(want < 152 * 16 ? want : 152 * 16);
  swa_to_bf16_kernel<<<grid, 256, 0, stream>>>(in, out, n8);
  return cudaGetLastError();
}

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t stream) {
  if (a.rows == 0) return cudaSuccess;
  const int DP = a.g.D <= 64 ? 64 : 128;
  const int64_t chunks = (a.rows + prep_chunk_rows(DP) - 1) / prep_chunk_rows(DP);
  const dim3 grid(static_cast<unsigned>(chunks));
  const size_t smem = prep_bulk_smem(DP);  // under the 48 KB a launch may use without opting in
  auto go = [&](auto kernel) { return launch_pdl(kernel, grid, dim3(kPrepThreads), smem, stream, a); };
  const bool exact = a.g.D == DP;
  if (DP == 64) {
    if (exact) return a.g.f16 ? go(swa_prep_bulk_kernel<64, true, true>) : go(swa_prep_bulk_kernel<64, false, true>);
    return a.g.f16 ? go(swa_prep_bulk_kernel<64, true, false>) : go(swa_prep_bulk_kernel<64, false, false>);
  }
  if (exact) return a.g.f16 ? go(swa_prep_bulk_kernel<128, true, true>) : go(swa_prep_bulk_kernel<128, false, true>);
  return a.g.f16 ? go(swa_prep_bulk_kernel<128, true, false>) : go(swa_prep_bulk_kernel<128, false, false>);
}

}  // namespace swa
