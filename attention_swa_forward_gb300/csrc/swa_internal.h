// swa_internal.h — shapes shared by the host scheduler and the kernels.
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "swa.h"

namespace swa {

constexpr int kTileM = 128;  // query rows per tile (tcgen05 M)
constexpr int kTileN = 128;  // key rows per tile

// One sequence of the batch as a kernel sees it.  BNSD: q_start = kv_start = 0
// (rows are addressed through b); TND: start rows inside [0, T).
struct SeqInfo {
  int32_t q_start, q_len, kv_start, kv_len;
  int64_t mask_base;  // dropout bit index of (n = 0, i = 0, j = 0) of this batch
};

// Work description passed to a kernel as a parameter (no device upload):
// a run of `heads * tiles` work items per entry.  A work item is one 128-row
// query tile (forward) or key tile (backward) of one (batch, head), numbered
// head by head (the tiles of one head are consecutive items, so the CTAs in
// flight share that head's tiles in L2).  For BNSD a single entry covers all
// B*N heads (b < 0; b = head / N); for TND each entry is one sequence (b >= 0;
// head = n).  Entries are ordered heaviest first and
// `descending` visits the tiles of an entry from the last one, so that the
// CTAs that start first carry the most work.
struct SeqDesc {
  int32_t q_start, q_len, kv_start, kv_len;
  int64_t mask_base;
  int32_t item_begin;  // first work item of this entry
  int32_t b;           // TND batch index, -1 for BNSD
  int32_t tiles;       // 128-row tiles per head
  int32_t heads;       // N (TND) or B*N (BNSD)
  int32_t descending;
  int32_t pad;
};
static_assert(sizeof(SeqDesc) == 48, "SeqDesc layout");

template <int CAP>
struct SeqTable {
  int32_t count;    // entries used
  int32_t n_items;  // work items of this launch
  int64_t pad;
  SeqDesc d[CAP];
};
constexpr int kSmallTable = 16;
constexpr int kLargeTable = 512;

// Workspace header (first 256 bytes of every workspace).
struct WsHeader {
  int32_t error;       // 0 = fine; otherwise the code of the wait that gave up
  int32_t pad[63];
};
constexpr size_t kHeaderBytes = 256;

// Raise a kernel's dynamic shared memory limit to `smem` bytes on the current
// device.  The setting belongs to the device's context, so it is made once
// per device (devices past 63 make it on every call); `done` is the kernel's
// own bit set, safe to share between host threads.
template <typename Kernel>
cudaError_t set_smem_limit(Kernel kernel, size_t smem, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// SWA_CHECKS = 1: the bounds-checked build (libswa_checked.so), whose kernels test every
// global load and store against its tensor's extent and record kErrBounds
// instead of making it.  Its host code clears the status word with a memset
// before a call's first launch, so that no grid's clear can race with a
// bounds record of another grid's block.
#ifndef SWA_CHECKS
#define SWA_CHECKS 0
#endif

// Error codes a kernel stores into WsHeader::error.
enum : int32_t {
  kErrFwdLoad = 1,
  kErrFwdMma = 2,
  kErrFwdSoftmax = 3,
  kErrBwdLoad = 11,
  kErrBwdMma = 12,
  kErrBwdCompute = 13,
  kErrPrepLoad = 14,  // the preprocess's wait for a chunk of dY / O
  kErrBounds = 21,  // bounds-checked build: an access outside its tensor was skipped
};

struct Geometry {
  int32_t layout;  // 0 = BNSD, 1 = TND
  int32_t N, D;
  int32_t N_kv;    // key/value heads; query head n reads key/value head n / group
  int32_t group;   // N / N_kv
  int32_t f16;     // element type of q, k, v, dy, out, dq, dk, dv: 0 bf16, 1 fp16
  int32_t S_q, S_kv;  // BNSD (per-batch lengths)
  int32_t sparse_mode;
  int32_t pre, next;  // clamped into +-(max sequence length + 1)
  float scale;        // score scale
  float scale_log2;   // scale * log2(e)
  float inv_keep;     // 1 / keep_prob
  float keep;         // keep_prob
  int32_t has_mask;   // dropout active (a drop_mask, or generated from seed / offset)
  int32_t drop_gen;   // 1: keep bits generated from (seed, offset) instead of read
  uint32_t seed_lo, seed_hi, off_lo;
  uint32_t keep_thr;  // element kept iff its Philox byte < keep_thr (0..256)
  int32_t T_q;        // query rows per head: B*S_q (BNSD) or T_q (TND)
  int32_t out_f32;    // outputs (out, dq, dk, dv) are fp32; the kernels then read bf16 copies of the inputs
  int32_t stall;      // test hook (swa_debug_stall): kStall* bits of kernels whose compute warps first wait
                      // on a barrier that nothing completes, so that the bounded wait runs out
  // Extents of the caller's tensors, which the bounds-checked build
  // (SWA_CHECKS = 1) tests every global access of the kernels against.
  int64_t n_q_elems;     // elements of q, dy, out and dq
  int64_t n_kv_elems;    // elements of k, v, dk and dv
  int64_t n_stats;       // query rows x heads: softmax_max, softmax_sum, lse2 and D entries
  int64_t n_mask_bytes;  // bytes of the packed keep mask (0 without one)
};

// Geometry::stall bits.
enum : int32_t { kStallForward = 1, kStallKeyMajor = 2, kStallQueryMajor = 4 };

struct FwdArgs {
  Geometry g;
  const uint8_t* mask;
  void* out;  // bf16 / fp16, or fp32 when g.out_f32
  float* smax;
  float* ssum;
  int32_t* err;
  int32_t clear_err;  // 1: block 0 clears *err on entry (the first launch of a forward call)
};

struct BwdArgs {
  Geometry g;
  const uint8_t* mask;
  const float* lse2;   // per query row, head-major (ws_stat_index): softmax_max*log2(e) + log2(softmax_sum); +inf for empty rows
  const float* dsum;   // per query row, head-major: D = rowsum(dY * O)
  void* dq;   // written by the query-major pass (element type as FwdArgs::out)
  void* dk;   // written by the key-major pass
  void* dv;
  int32_t* err;
};

struct PrepArgs {
  Geometry g;
  int64_t rows;  // query rows x heads
  int32_t* err;  // workspace error word, cleared here before the backward kernel runs
  const __nv_bfloat16* dy;
  const __nv_bfloat16* out;
  const float* smax;
  const float* ssum;
  float* lse2;
  float* dsum;
};

// Dropout mode DM: 0 none, 1 keep bits read from the caller's mask, 2 keep
// bits generated from (seed, offset).
__host__ __device__ constexpr int drop_mode_of(int has_mask, int gen) { return has_mask ? (gen ? 2 : 1) : 0; }

// Record `fmt` as the text of swa_last_error() on this thread; returns st.
swa_status_t set_error(swa_status_t st, const char* fmt, ...);

// Kernel launchers (defined in the .cu files).  Each returns the launch's
// cudaError_t.
template <int CAP>
cudaError_t launch_forward(const FwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq, const CUtensorMap& mk,
                           const CUtensorMap& mv, cudaStream_t stream);
// D <= 64: one CTA per pair of query tiles; the table's entries count pairs
// (tiles = ceil(query tiles / 2)).
template <int CAP>
cudaError_t launch_forward_pair(const FwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq,
                                const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t stream);
template <int CAP>
cudaError_t launch_backward_dkv(const BwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq,
                                const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdy,
                                cudaStream_t stream);
template <int CAP>
cudaError_t launch_backward_dq(const BwdArgs& a, const SeqTable<CAP>& tab, const CUtensorMap& mq,
                               const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdy,
                               cudaStream_t stream);
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t stream);
// fp32 -> bf16 (round to nearest even) of n elements, n a multiple of 8, both 16-byte aligned.
cudaError_t launch_to_bf16(const float* in, __nv_bfloat16* out, int64_t n, cudaStream_t stream);

// The packed keep mask a seed / offset pair stands for: one CTA per query
// tile of a (batch, head) from the forward's work table, one thread per
// query row; bits are OR-ed into the zeroed mask.
struct MaskGenArgs {
  Geometry g;
  uint32_t* mask;  // 32-bit words of the packed mask, zeroed beforehand
};
template <int CAP>
cudaError_t launch_dropout_mask(const MaskGenArgs& a, const SeqTable<CAP>& tab, cudaStream_t stream);

}  // namespace swa
