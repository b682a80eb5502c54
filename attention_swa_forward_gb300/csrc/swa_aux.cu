// swa_aux.cu — the memory-bound pass before the backward kernels.
//
//  * preprocess: per query row, D = rowsum(dY * O) (PyPTO-Gym article,
//    "反向公式") and lse2 = softmax_max*log2(e) + log2(softmax_sum) (+inf for
//    an empty row, so that the recomputed P is 0).
//
// Both layouts address a query row (b, n, i) / (t, n) the same way once
// flattened: row id r -> elements [r*D, r*D + D), statistics index r.
#include "swa_internal.h"
#include "sm103.cuh"

namespace swa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// One warp per row; each lane handles D/32 consecutive elements.
template <int D>
__global__ void __launch_bounds__(256) swa_prep_kernel(const PrepArgs a) {
  constexpr int kPer = D / 32;  // 2 or 4 bf16 per lane
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.err = 0;  // fresh error word for this backward call
  if (row >= a.rows) return;
  const int64_t base = row * D + lane * kPer;
  float acc = 0.f;
  if (kPer == 4) {
    const uint2 dy = __ldg(reinterpret_cast<const uint2*>(a.dy + base));
    const uint2 o = __ldg(reinterpret_cast<const uint2*>(a.out + base));
    const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dy);
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const float2 df = __bfloat1622float2(d2[t]);
      const float2 of = __bfloat1622float2(o2[t]);
      acc = fmaf(df.x, of.x, acc);
      acc = fmaf(df.y, of.y, acc);
    }
  } else {
    const uint32_t dy = __ldg(reinterpret_cast<const uint32_t*>(a.dy + base));
    const uint32_t o = __ldg(reinterpret_cast<const uint32_t*>(a.out + base));
    const float2 df = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dy));
    const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o));
    acc = fmaf(df.x, of.x, acc);
    acc = fmaf(df.y, of.y, acc);
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, m);
  if (lane == 0) {
    const float l = a.ssum[row];
    a.dsum[row] = acc;
    a.lse2[row] = (l > 0.f) ? a.smax[row] * kLog2e + __log2f(l) : INFINITY;
  }
}

}  // namespace

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t stream) {
  if (a.rows == 0) return cudaSuccess;
  const int64_t threads = a.rows * 32;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  if (a.g.D == 64)
    swa_prep_kernel<64><<<static_cast<unsigned>(grid), block, 0, stream>>>(a);
  else
    swa_prep_kernel<128><<<static_cast<unsigned>(grid), block, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace swa
