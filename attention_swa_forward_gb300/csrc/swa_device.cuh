// swa_device.cuh — device helpers shared by the forward and backward kernels:
// addressing of BNSD / TND rows, the BAND window, tile loads, dropout bits and
// writing a bf16 row into a 128-byte-swizzled shared-memory tile.
#pragma once
#include <utility>

#include "sm103.cuh"
#include "swa_internal.h"
#include "swa_sched.h"

namespace swa {

constexpr int kAtomBytes = 128 * 128;  // one atom column: 128 rows x 128 bytes

// Launch with programmatic stream serialization: the kernel may start while
// the previous grid on the stream finishes; it calls griddep_wait before
// reading what that grid (or an earlier one) wrote.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Element offset of local query row i of (b, n): BNSD [B,N,S,D] or TND [T,N,D].
__device__ __forceinline__ int64_t q_elem(const Geometry& g, const SeqInfo& s, int b, int n, int i) {
  return g.layout == 0 ? ((static_cast<int64_t>(b) * g.N + n) * g.S_q + i) * g.D
                       : (static_cast<int64_t>(s.q_start + i) * g.N + n) * g.D;
}
// Element offset of local key row j of key/value head h: BNSD [B,N_kv,S,D] or TND [T,N_kv,D].
__device__ __forceinline__ int64_t kv_elem(const Geometry& g, const SeqInfo& s, int b, int h, int j) {
  return g.layout == 0 ? ((static_cast<int64_t>(b) * g.N_kv + h) * g.S_kv + j) * g.D
                       : (static_cast<int64_t>(s.kv_start + j) * g.N_kv + h) * g.D;
}
// Index of the softmax statistics of local query row i: [B,N,S] or [T,N].
__device__ __forceinline__ int64_t stat_index(const Geometry& g, const SeqInfo& s, int b, int n, int i) {
  return g.layout == 0 ? (static_cast<int64_t>(b) * g.N + n) * g.S_q + i
                       : static_cast<int64_t>(s.q_start + i) * g.N + n;
}

// Position of local query row i of head n in the backward workspace's lse2 /
// D arrays: head-major in both layouts ([B,N,S] for BNSD, [N,T] for TND), so
// that the 128 rows of one head in a query tile are contiguous (in the [T,N]
// order of the statistics they would be N elements apart, one cache line each).
__device__ __forceinline__ int64_t ws_stat_index(const Geometry& g, const SeqInfo& s, int b, int n, int i) {
  return g.layout == 0 ? (static_cast<int64_t>(b) * g.N + n) * g.S_q + i
                       : static_cast<int64_t>(n) * g.T_q + (s.q_start + i);
}

// Keys visible to local query row i: [lo, hi] (empty when lo > hi).
// sparse_mode 4 (BAND): i - pre <= j <= i + next; rows past the sequence see nothing.
__device__ __forceinline__ void key_window(const Geometry& g, const SeqInfo& s, int i, int& lo, int& hi) {
  lo = 0;
  hi = s.kv_len - 1;
  if (g.sparse_mode == 4) {
    lo = max(lo, i - g.pre);
    hi = min(hi, i + g.next);
  }
  if (i >= s.q_len) {
    lo = 1;
    hi = 0;
  }
}

// 16-column steps of a contraction over the head dim: the kernels hold 64 or
// 128 columns per row, and the columns past D (zero-filled by the tensor map)
// add nothing, so the steps past them are skipped.
__device__ __forceinline__ int d_steps(const Geometry& g) { return (g.D + 15) >> 4; }

// Is every (i, j) of the query tile [q0, q0+128) x key tile [j0, j0+128) visible?
__device__ __forceinline__ bool tile_fully_visible(const Geometry& g, const SeqInfo& s, int q0, int j0) {
  if (q0 + 127 >= s.q_len || j0 + 127 >= s.kv_len) return false;
  if (g.sparse_mode != 4) return true;
  return j0 >= q0 + 127 - g.pre && j0 + 127 <= q0 + g.next;
}

// TMA load of 128 rows x D columns starting at local row `row0` of (b, n) into
// D/64 consecutive atom columns.  BNSD maps are (d, s, n, b); TND maps are
// (d, n, t, 1) and take the sequence's start row.
template <int D>
__device__ __forceinline__ void tma_rows(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, const Geometry& g,
                                         int b, int n, int start, int row0) {
#pragma unroll
  for (int a = 0; a < D / 64; ++a) {
    if (g.layout == 0)
      tma_load_4d(dst + a * kAtomBytes, map, bar, a * 64, row0, n, b);
    else
      tma_load_4d(dst + a * kAtomBytes, map, bar, a * 64, n, start + row0, 0);
  }
}

// --------------------------------------------------- bounds-checked build --
// Built with SWA_CHECKS = 1, the kernels test every global load and store
// against the extent of its tensor first (Geometry::n_*): an access outside
// it is skipped and kErrBounds recorded in the status word, so an indexing
// or scheduling error shows up as a status instead of as a memory fault.
// The release build compiles the tests away.  (Tiled TMA copies need no
// test: the tensor maps bound them.  The preprocess's untiled bulk copies
// are tested.)  SWA_CHECKS itself is set in swa_internal.h.
__device__ __forceinline__ bool in_bounds(int64_t first, int64_t count, int64_t extent, int32_t* err) {
  if constexpr (SWA_CHECKS == 0) {
    return true;
  } else {
    if (first >= 0 && count >= 0 && first + count <= extent) return true;
    atomicCAS(err, 0, static_cast<int32_t>(kErrBounds));
    return false;
  }
}

// 128 dropout keep bits of row i for keys [j0, j0+128): bit t of the result
// (word t >> 5) is key j0 + t.  Bits past the sequence's last key are 0.
// Element order: mask_base + (n*Sq + i)*Skv + j, least significant bit first.
// `extent` (mask bytes) and `err` serve the bounds-checked build.
__device__ __forceinline__ void load_keep_bits(const uint8_t* __restrict__ mask, const SeqInfo& s, int n, int i,
                                               int j0, uint32_t (&bits)[4], int64_t extent, int32_t* err) {
  const int cnt = min(128, s.kv_len - j0);
  const int64_t e0 = s.mask_base + (static_cast<int64_t>(n) * s.q_len + i) * s.kv_len + j0;
  uint32_t w[5] = {0u, 0u, 0u, 0u, 0u};
  const int sh = static_cast<int>(e0 & 7);
  const uint8_t* p = mask + (e0 >> 3);
  const bool whole = (e0 & 127) == 0 && cnt == 128;
  if (!in_bounds(e0 >> 3, whole ? 16 : (sh + cnt + 7) >> 3, extent, err)) {
#pragma unroll
    for (int k = 0; k < 4; ++k) bits[k] = 0u;
    return;
  }
  if (whole) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    const int nbytes = (sh + cnt + 7) >> 3;
#pragma unroll
    for (int t = 0; t < 17; ++t)
      if (t < nbytes) w[t >> 2] |= static_cast<uint32_t>(__ldg(p + t)) << ((t & 3) * 8);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) bits[k] = __funnelshift_r(w[k], w[k + 1], sh);
  if (cnt < 128) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int lo = k * 32;
      const uint32_t keep = cnt >= lo + 32 ? 0xFFFFFFFFu : (cnt <= lo ? 0u : ((1u << (cnt - lo)) - 1u));
      bits[k] &= keep;
    }
  }
}

// ------------------------------------------------- generated keep bits --
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11): ten rounds; each multiplies counter words 0 and 2
// by 0xD2511F53 and 0xCD9E8D57 (32x32 -> 64 bits) and forms the new counter
// (hi(c2*M1) ^ c1 ^ k0, lo(c2*M1), hi(c0*M0) ^ c3 ^ k1, lo(c0*M0)); the key
// is bumped by (0x9E3779B9, 0xBB67AE85) after every round.
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                               uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return make_uint4(c0, c1, c2, c3);
}

// Bit m (0..3) set iff byte m of w is below thr (thr in 0..256).
__device__ __forceinline__ uint32_t keep4(uint32_t w, uint32_t thr) {
  if (thr >= 256u) return 0xFu;
  const uint32_t m = __vcmpltu4(w, thr * 0x01010101u) & 0x01010101u;  // 1 per kept byte
  return (m * 0x10204080u) >> 28;  // gathers the four byte flags into bits 28..31
}

// Keep bits of query row `row` (its statistics id) for local keys
// [16*kb, 16*kb + 16): bit m is key 16*kb + m.  The element is kept iff byte
// (j mod 16) of Philox4x32-10(counter = (j/16, lo32 row, hi32 row, lo32
// offset), key = seed) is below keep_thr, bytes little-endian across the
// four output words.
__device__ __forceinline__ uint32_t gen_keep16(const Geometry& g, int64_t row, int kb) {
  const uint4 r = philox4x32_10(static_cast<uint32_t>(kb), static_cast<uint32_t>(row),
                                static_cast<uint32_t>(static_cast<uint64_t>(row) >> 32), g.off_lo, g.seed_lo,
                                g.seed_hi);
  return keep4(r.x, g.keep_thr) | (keep4(r.y, g.keep_thr) << 4) | (keep4(r.z, g.keep_thr) << 8) |
         (keep4(r.w, g.keep_thr) << 12);
}

// NW 32-bit keep words of row `row` for local keys [16*kb0, 16*kb0 + 32*NW):
// bit t of word t>>5 is key 16*kb0 + t (the layout load_keep_bits returns).
template <int NW>
__device__ __forceinline__ void gen_keep_words(const Geometry& g, int64_t row, int kb0, uint32_t* words) {
#pragma unroll
  for (int q = 0; q < NW; ++q) words[q] = gen_keep16(g, row, kb0 + 2 * q) | (gen_keep16(g, row, kb0 + 2 * q + 1) << 16);
}

// Write 8 bf16 (one 16-byte chunk) of row r, chunk index c (0..15 over a
// 128-wide row spanning two atom columns) into a swizzled tile.
__device__ __forceinline__ void st_chunk_sw128(uint8_t* tile, int r, int c, uint4 v) {
  uint8_t* dst = tile + (c >> 3) * kAtomBytes + r * 128 + ((((c & 7) ^ r) & 7) << 4);
  *reinterpret_cast<uint4*>(dst) = v;
}

__device__ __forceinline__ uint4 ld_chunk_sw128(const uint8_t* tile, int r, int c) {
  return *reinterpret_cast<const uint4*>(tile + (c >> 3) * kAtomBytes + r * 128 + ((((c & 7) ^ r) & 7) << 4));
}

// x where bit b of w is set, +0 where it is clear: the bit, moved to the
// sign position and sign-extended, masks x (no predicate, no select).
__device__ __forceinline__ float keep_or_zero(float x, uint32_t w, int b) {
  const uint32_t m = static_cast<uint32_t>(static_cast<int32_t>(w << (31 - b)) >> 31);
  return __uint_as_float(__float_as_uint(x) & m);
}

// 32 x 32 bit-matrix transpose across a warp (all 32 lanes converged).  On
// entry lane l holds row l of the matrix (bit k = element (l, k)); on exit
// lane k holds column k (bit l = element (l, k)).  Transposing swaps each bit
// of the row index with the same bit of the column index; stage j swaps bit j,
// which trades the two off-diagonal j x j blocks of every 2j x 2j block
// between lane pairs l, l ^ j.
__device__ __forceinline__ uint32_t warp_transpose_bits(uint32_t x, int lane) {
  constexpr uint32_t kLowCols[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int s = 0; s < 5; ++s) {
    const int j = 16 >> s;
    const uint32_t m = kLowCols[s];  // the columns whose bit j is clear
    const uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, x, j);
    x = (lane & j) ? ((x & ~m) | ((y >> j) & m)) : ((x & m) | ((y << j) & ~m));
  }
  return x;
}

template <bool F16>
__device__ __forceinline__ uint4 pack8(const float* x) {
  uint4 v;
  v.x = pack2<F16>(x[0], x[1]);
  v.y = pack2<F16>(x[2], x[3]);
  v.z = pack2<F16>(x[4], x[5]);
  v.w = pack2<F16>(x[6], x[7]);
  return v;
}

// Eight consecutive output elements from element e of `base` on: packed to
// the element type (bf16 / fp16), or stored as fp32 when `f32`.  e is a
// multiple of 8, so both forms are 16-byte aligned.
template <bool F16>
__device__ __forceinline__ void store8(void* base, int64_t e, const float* x, bool f32) {
  if (f32) {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(base) + e);
    d[0] = make_float4(x[0], x[1], x[2], x[3]);
    d[1] = make_float4(x[4], x[5], x[6], x[7]);
  } else {
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + e) = pack8<F16>(x);
  }
}

}  // namespace swa
