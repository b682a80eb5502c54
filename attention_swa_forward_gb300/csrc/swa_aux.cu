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

// One warp per row; each lane handles DP/32 consecutive elements of a row of
// D <= DP elements (D a multiple of 8: a lane's elements lie all below D or
// all past it).
template <int DP, bool F16>
__global__ void __launch_bounds__(256) swa_prep_kernel(const PrepArgs a) {
  constexpr int kPer = DP / 32;  // 2 or 4 elements per lane
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  griddep_wait();  // dY, O and the statistics come from earlier grids
  griddep_launch_dependents();
  if (!SWA_CHECKS && blockIdx.x == 0 && threadIdx.x == 0) *a.err = 0;  // fresh error word for this backward call
  if (row >= a.rows) return;
  const int D = a.g.D;
  const int64_t base = row * D + lane * kPer;
  float acc = 0.f;
  if (lane * kPer >= D || !in_bounds(base, kPer, a.g.n_q_elems, a.err)) {
    // past the row's last element
  } else if (kPer == 4) {
    const uint2 dy = __ldg(reinterpret_cast<const uint2*>(a.dy + base));
    const uint2 o = __ldg(reinterpret_cast<const uint2*>(a.out + base));
    const uint32_t d2[2] = {dy.x, dy.y}, o2[2] = {o.x, o.y};
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const float2 df = unpack2<F16>(d2[t]);
      const float2 of = unpack2<F16>(o2[t]);
      acc = fmaf(df.x, of.x, acc);
      acc = fmaf(df.y, of.y, acc);
    }
  } else {
    const uint32_t dy = __ldg(reinterpret_cast<const uint32_t*>(a.dy + base));
    const uint32_t o = __ldg(reinterpret_cast<const uint32_t*>(a.out + base));
    const float2 df = unpack2<F16>(dy);
    const float2 of = unpack2<F16>(o);
    acc = fmaf(df.x, of.x, acc);
    acc = fmaf(df.y, of.y, acc);
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, m);
  if (lane == 0) {
    // workspace position: head-major (row = t*N + n in TND, already head-major in BNSD)
    const int64_t ws = a.g.layout == 0 ? row : (row % a.g.N) * a.g.T_q + row / a.g.N;
    if (!in_bounds(row, 1, a.g.n_stats, a.err) || !in_bounds(ws, 1, a.g.n_stats, a.err)) return;
    const float l = a.ssum[row];
    a.dsum[ws] = acc;
    a.lse2[ws] = (l > 0.f) ? a.smax[row] * kLog2e + __log2f(l) : INFINITY;
  }
}

// The same for D = 64 or 128 exactly, with more bytes in flight: a row is
// split over D/8 lanes (16 bytes of dY and of O each), a warp covers 32/(D/8)
// rows per load step and kSteps steps, all loads issued before any use.  The
// kernel is memory-latency bound (its loads in flight per SM set the rate),
// so it is held to 64 registers a thread, which fits four blocks of 256
// threads per SM instead of three: 0.70 -> 0.79 of the measured copy
// bandwidth on 32 x 32768 rows of D = 128 (0.117 -> 0.103 ms).
template <int D, bool F16>
__global__ void __launch_bounds__(256, 4) swa_prep_wide_kernel(const PrepArgs a) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerStep = 32 / kLanesPerRow;
  constexpr int kSteps = 4;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  griddep_wait();  // dY, O and the statistics come from earlier grids
  griddep_launch_dependents();
  if (!SWA_CHECKS && blockIdx.x == 0 && threadIdx.x == 0) *a.err = 0;  // fresh error word for this backward call
  const int64_t row0 = warp * (kRowsPerStep * kSteps) + lane / kLanesPerRow;
  const int col = (lane % kLanesPerRow) * 8;
  // row r of step k is row0 + k * kRowsPerStep: one base pointer per tensor
  // and a fixed stride, so the addresses cost one add per load
  const uint4* pdy = reinterpret_cast<const uint4*>(a.dy + row0 * D + col);
  const uint4* po = reinterpret_cast<const uint4*>(a.out + row0 * D + col);
  constexpr int kStride = kRowsPerStep * D / 8;  // uint4 per step
  const int64_t left = a.rows > row0 ? (a.rows - row0 + kRowsPerStep - 1) / kRowsPerStep : 0;
  const int nvalid = left < kSteps ? static_cast<int>(left) : kSteps;  // steps whose row exists
  uint4 dy[kSteps], o[kSteps];
#pragma unroll
  for (int k = 0; k < kSteps; ++k) {
    if (k < nvalid && in_bounds((row0 + k * kRowsPerStep) * D + col, 8, a.g.n_q_elems, a.err)) {
      dy[k] = __ldg(pdy + k * kStride);
      o[k] = __ldg(po + k * kStride);
    } else {
      dy[k] = o[k] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int k = 0; k < kSteps; ++k) {
    const uint32_t d4[4] = {dy[k].x, dy[k].y, dy[k].z, dy[k].w}, o4[4] = {o[k].x, o[k].y, o[k].z, o[k].w};
    float acc = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 df = unpack2<F16>(d4[t]), of = unpack2<F16>(o4[t]);
      acc = fmaf(df.x, of.x, acc);
      acc = fmaf(df.y, of.y, acc);
    }
#pragma unroll
    for (int m = kLanesPerRow / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, m);
    const int64_t row = row0 + k * kRowsPerStep;
    if (lane % kLanesPerRow == 0 && k < nvalid) {
      const int64_t ws = a.g.layout == 0 ? row : (row % a.g.N) * a.g.T_q + row / a.g.N;
      if (!in_bounds(row, 1, a.g.n_stats, a.err) || !in_bounds(ws, 1, a.g.n_stats, a.err)) continue;
      const float l = a.ssum[row];
      a.dsum[ws] = acc;
      a.lse2[ws] = (l > 0.f) ? a.smax[row] * kLog2e + __log2f(l) : INFINITY;
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
  if (a.g.D == 64 || a.g.D == 128) {
    const int64_t rows_per_block = 8 * (32 / (a.g.D / 8)) * 4;  // 8 warps x rows per step x 4 steps
    const unsigned gr = static_cast<unsigned>((a.rows + rows_per_block - 1) / rows_per_block);
    if (a.g.D == 64) {
      if (a.g.f16) return launch_pdl(swa_prep_wide_kernel<64, true>, dim3(gr), dim3(256), 0, stream, a);
      return launch_pdl(swa_prep_wide_kernel<64, false>, dim3(gr), dim3(256), 0, stream, a);
    } else {
      if (a.g.f16) return launch_pdl(swa_prep_wide_kernel<128, true>, dim3(gr), dim3(256), 0, stream, a);
      return launch_pdl(swa_prep_wide_kernel<128, false>, dim3(gr), dim3(256), 0, stream, a);
    }
  }
  const int64_t threads = a.rows * 32;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  const unsigned gr = static_cast<unsigned>(grid);
  if (a.g.D <= 64) {
    if (a.g.f16) return launch_pdl(swa_prep_kernel<64, true>, dim3(gr), dim3(block), 0, stream, a);
    return launch_pdl(swa_prep_kernel<64, false>, dim3(gr), dim3(block), 0, stream, a);
  } else {
    if (a.g.f16) return launch_pdl(swa_prep_kernel<128, true>, dim3(gr), dim3(block), 0, stream, a);
    return launch_pdl(swa_prep_kernel<128, false>, dim3(gr), dim3(block), 0, stream, a);
  }
  return cudaGetLastError();
}

}  // namespace swa
