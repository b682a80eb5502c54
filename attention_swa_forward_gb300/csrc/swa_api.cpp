// swa_api.cpp — the C ABI of libswa (include/swa.h): argument checks, the
// band / varlen tile scheduler, TMA descriptors and kernel launches.
//
// Follows the two-phase workspace convention and status codes of the
// FlashAttentionVarLenScore doc ("两段式接口", "返回值"), and the swa_forward /
// swa_backward split limited to sparse modes 0 and 4 (pzsr.cn article §3).
#include "swa.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include "swa_internal.h"
#include "swa_sched.h"

using namespace swa;

namespace {

thread_local std::string t_last_error = "no error";
std::atomic<int32_t> g_stall{0};  // swa_debug_stall: read into Geometry::stall by every call
std::atomic<int32_t> g_fwd_pairs{0};  // swa_debug_forward_pairs: 0 by size, 1 always, 2 never
std::atomic<int64_t> g_extent_slack{0};  // swa_debug_extent_slack: taken off every extent of the bounds checks
thread_local cudaEvent_t t_ev[8] = {};  // start/stop around: forward, dK/dV pass, dQ pass, preprocess

swa_status_t fail(swa_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

constexpr int64_t kMaxRows = int64_t(1) << 20;  // T (TND) or S (BNSD) limit: 1M rows
constexpr double kLog2e = 1.4426950408889634;

struct Seq {
  int64_t q_start, q_len, kv_start, kv_len, mask_base;
};

struct Plan {
  Geometry g{};
  int64_t B = 0;
  std::vector<Seq> seqs;       // per batch
  int64_t q_rows = 0;          // rows of q per head: B*S_q or T_q
  int64_t kv_rows = 0;
  int64_t mask_bits = 0;
};

// Sequence spans from cumulative ends; a drop (trailing zeros) marks skipped
// batches (aclnnFlashAttentionUnpaddingScoreGradV2 article §6.4).
swa_status_t parse_cumulative(const int64_t* cu, int64_t B, int64_t T, const char* name, std::vector<int64_t>& start,
                              std::vector<int64_t>& len) {
  start.assign(B, 0);
  len.assign(B, 0);
  int64_t prev = 0;
  bool in_tail = false;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t e = cu[b];
    if (in_tail) {
      if (e != 0) return fail(SWA_ERR_PARAM_INVALID, "%s[%lld] = %lld after the trailing zeros", name, (long long)b,
                              (long long)e);
      start[b] = T;
      continue;
    }
    if (e < prev) {
      if (e != 0) return fail(SWA_ERR_PARAM_INVALID, "%s is not non-decreasing at index %lld", name, (long long)b);
      if (prev != T) return fail(SWA_ERR_PARAM_INVALID, "%s ends at %lld before its trailing zeros, T = %lld", name,
                                 (long long)prev, (long long)T);
      in_tail = true;
      start[b] = T;
      continue;
    }
    start[b] = prev;
    len[b] = e - prev;
    prev = e;
  }
  if (!in_tail && prev != T)
    return fail(SWA_ERR_PARAM_INVALID, "%s ends at %lld but T = %lld", name, (long long)prev, (long long)T);
  return SWA_OK;
}

swa_status_t make_plan(const swa_params_t* p, Plan& plan) {
  if (!p) return fail(SWA_ERR_PARAM_NULLPTR, "params is NULL");
  if (p->layout != SWA_LAYOUT_BNSD && p->layout != SWA_LAYOUT_TND)
    return fail(SWA_ERR_PARAM_INVALID, "layout %d is neither BNSD (0) nor TND (1)", p->layout);
  if (p->sparse_mode != 0 && p->sparse_mode != 4)
    return fail(SWA_ERR_PARAM_INVALID, "sparse_mode should be 0 or 4, got %d", p->sparse_mode);
  if (!(p->keep_prob > 0.0 && p->keep_prob <= 1.0))
    return fail(SWA_ERR_PARAM_INVALID, "keep_prob must be in (0, 1], got %g", p->keep_prob);
  if (p->N < 1 || p->N > 256) return fail(SWA_ERR_PARAM_INVALID, "N must be in [1, 256], got %lld", (long long)p->N);
  const int64_t n_kv = p->N_kv == 0 ? p->N : p->N_kv;
  if (n_kv < 1 || n_kv > p->N || p->N % n_kv != 0)
    return fail(SWA_ERR_PARAM_INVALID, "N = %lld must be a multiple of N_kv = %lld", (long long)p->N,
                (long long)p->N_kv);
  if (p->B < 1) return fail(SWA_ERR_PARAM_INVALID, "B must be >= 1, got %lld", (long long)p->B);
  if (p->D < 1 || p->D > 768) return fail(SWA_ERR_PARAM_INVALID, "D must be in [1, 768], got %lld", (long long)p->D);
  // D up to 128 in steps of 8 (a row then starts on a 16-byte boundary, as a
  // TMA copy needs); the kernels compute on 64 or 128 columns and the tensor
  // maps fill the columns past D with zeros.
  if (p->D % 8 != 0 || p->D > 128)
    return fail(SWA_ERR_UNSUPPORTED, "D = %lld is not built (a multiple of 8 up to 128)", (long long)p->D);
  if (!std::isfinite(p->scale)) return fail(SWA_ERR_PARAM_INVALID, "scale is not finite");
  if (p->sparse_mode == 4) {
    // an everywhere-empty band is almost certainly a caller error
    const long double s = (long double)p->pre_tokens + (long double)p->next_tokens;
    if (s < 0) return fail(SWA_ERR_PARAM_INVALID, "pre_tokens + next_tokens < 0: every row would be empty");
  }

  plan = Plan();
  plan.B = p->B;
  Geometry& g = plan.g;
  g.layout = p->layout;
  g.N = static_cast<int32_t>(p->N);
  g.N_kv = static_cast<int32_t>(n_kv);
  g.group = static_cast<int32_t>(p->N / n_kv);
  g.D = static_cast<int32_t>(p->D);
  g.sparse_mode = p->sparse_mode;
  g.scale = static_cast<float>(p->scale);
  g.scale_log2 = static_cast<float>(p->scale * kLog2e);
  g.inv_keep = static_cast<float>(1.0 / p->keep_prob);
  g.keep = static_cast<float>(p->keep_prob);
  if (p->dtype != SWA_DTYPE_BF16 && p->dtype != SWA_DTYPE_FP16 && p->dtype != SWA_DTYPE_FP32)
    return fail(SWA_ERR_PARAM_INVALID, "dtype should be 0 (bf16), 1 (fp16) or 2 (fp32), got %d", p->dtype);
  // fp32: the kernels run on bf16 copies of the inputs made in the workspace
  // and store fp32 outputs
  g.f16 = p->dtype == SWA_DTYPE_FP16 ? 1 : 0;
  g.out_f32 = p->dtype == SWA_DTYPE_FP32 ? 1 : 0;
  if (p->dropout_gen != 0 && p->dropout_gen != 1)
    return fail(SWA_ERR_PARAM_INVALID, "dropout_gen should be 0 or 1, got %d", p->dropout_gen);
  g.has_mask = p->keep_prob < 1.0;
  g.drop_gen = (p->dropout_gen == 1 && p->keep_prob < 1.0) ? 1 : 0;
  g.seed_lo = static_cast<uint32_t>(p->dropout_seed);
  g.seed_hi = static_cast<uint32_t>(p->dropout_seed >> 32);
  g.off_lo = static_cast<uint32_t>(p->dropout_offset);
  g.keep_thr = static_cast<uint32_t>(std::min(256L, std::max(0L, std::lround(p->keep_prob * 256.0))));
  g.stall = g_stall.load(std::memory_order_relaxed);

  int64_t max_len = 0;
  if (p->layout == SWA_LAYOUT_BNSD) {
    if (p->S_q < 1 || p->S_q > kMaxRows || p->S_kv < 1 || p->S_kv > kMaxRows)
      return fail(SWA_ERR_PARAM_INVALID, "S_q / S_kv must be in [1, %lld]", (long long)kMaxRows);
    if (p->B * p->S_q > (int64_t(1) << 31) || p->B * p->S_kv > (int64_t(1) << 31))
      return fail(SWA_ERR_PARAM_INVALID, "B * S exceeds 2^31 rows");
    g.S_q = static_cast<int32_t>(p->S_q);
    g.S_kv = static_cast<int32_t>(p->S_kv);
    plan.seqs.resize(p->B);
    for (int64_t b = 0; b < p->B; ++b)
      plan.seqs[b] = Seq{0, p->S_q, 0, p->S_kv, b * p->N * p->S_q * p->S_kv};
    plan.q_rows = p->B * p->S_q;
    g.T_q = static_cast<int32_t>(plan.q_rows);
    plan.kv_rows = p->B * p->S_kv;
    plan.mask_bits = p->B * p->N * p->S_q * p->S_kv;
    max_len = std::max(p->S_q, p->S_kv);
  } else {
    if (!p->cu_seqlens_q || !p->cu_seqlens_kv) return fail(SWA_ERR_PARAM_NULLPTR, "cu_seqlens_q / cu_seqlens_kv is NULL");
    if (p->T_q < 1 || p->T_q > kMaxRows || p->T_kv < 1 || p->T_kv > kMaxRows)
      return fail(SWA_ERR_PARAM_INVALID, "T_q / T_kv must be in [1, %lld]", (long long)kMaxRows);
    std::vector<int64_t> qs, ql, ks, kl;
    swa_status_t st = parse_cumulative(p->cu_seqlens_q, p->B, p->T_q, "cu_seqlens_q", qs, ql);
    if (st != SWA_OK) return st;
    st = parse_cumulative(p->cu_seqlens_kv, p->B, p->T_kv, "cu_seqlens_kv", ks, kl);
    if (st != SWA_OK) return st;
    plan.seqs.resize(p->B);
    int64_t bits = 0;
    for (int64_t b = 0; b < p->B; ++b) {
      plan.seqs[b] = Seq{qs[b], ql[b], ks[b], kl[b], bits};
      bits += p->N * ql[b] * kl[b];
      max_len = std::max(max_len, std::max(ql[b], kl[b]));
    }
    g.S_q = 0;
    g.S_kv = 0;
    plan.q_rows = p->T_q;
    g.T_q = static_cast<int32_t>(plan.q_rows);
    plan.kv_rows = p->T_kv;
    plan.mask_bits = bits;
  }
  // tensor extents, for the bounds-checked build's device-side checks
  g.n_q_elems = plan.q_rows * p->N * p->D;
  g.n_kv_elems = plan.kv_rows * g.N_kv * p->D;
  g.n_stats = plan.q_rows * p->N;
  g.n_mask_bytes = (g.has_mask && !g.drop_gen) ? (plan.mask_bits + 7) / 8 : 0;
  const int64_t slack = g_extent_slack.load(std::memory_order_relaxed);
  for (int64_t* x : {&g.n_q_elems, &g.n_kv_elems, &g.n_stats, &g.n_mask_bytes}) *x = std::max<int64_t>(*x - slack, 0);
  // The window cannot reach further than the longest sequence: clamp.
  const int64_t lim = max_len + 1;
  g.pre = static_cast<int32_t>(std::min(std::max(p->pre_tokens, -lim), lim));
  g.next = static_cast<int32_t>(std::min(std::max(p->next_tokens, -lim), lim));
  return SWA_OK;
}

// ------------------------------------------------------------ scheduler --
SeqInfo info_of(const Seq& s) {
  SeqInfo x{};
  x.q_start = static_cast<int32_t>(s.q_start);
  x.q_len = static_cast<int32_t>(s.q_len);
  x.kv_start = static_cast<int32_t>(s.kv_start);
  x.kv_len = static_cast<int32_t>(s.kv_len);
  x.mask_base = s.mask_base;
  return x;
}
// Number of key tiles a query tile visits (forward, query-major pass) or
// query tiles a key tile visits (key-major pass): the kernels' own ranges.
int64_t fwd_tile_cost(const Geometry& g, const Seq& s, int64_t t) {
  int t0, n;
  key_tiles_of_query_tile(g, info_of(s), static_cast<int>(t), &t0, &n);
  return n;
}
int64_t bwd_tile_cost(const Geometry& g, const Seq& s, int64_t t) {
  int t0, n;
  query_tiles_of_key_tile(g, info_of(s), static_cast<int>(t), &t0, &n);
  return n;
}

// Work entries of one launch family, heaviest first.
std::vector<SeqDesc> build_descs(const Plan& plan, bool forward) {
  const Geometry& g = plan.g;
  struct Entry {
    SeqDesc d;
    int64_t weight;
  };
  std::vector<Entry> entries;
  auto fill = [&](const Seq& s, int32_t b, int32_t heads) {
    const int64_t rows = forward ? s.q_len : s.kv_len;
    if (rows <= 0) return;
    const int64_t tiles = (rows + kTileM - 1) / kTileM;
    int64_t wmax = 0;
    for (int64_t t = 0; t < tiles; ++t)
      wmax = std::max(wmax, forward ? fwd_tile_cost(g, s, t) : bwd_tile_cost(g, s, t));
    const int64_t c0 = forward ? fwd_tile_cost(g, s, 0) : bwd_tile_cost(g, s, 0);
    const int64_t c1 = forward ? fwd_tile_cost(g, s, tiles - 1) : bwd_tile_cost(g, s, tiles - 1);
    SeqDesc d{};
    d.q_start = static_cast<int32_t>(s.q_start);
    d.q_len = static_cast<int32_t>(s.q_len);
    d.kv_start = static_cast<int32_t>(s.kv_start);
    d.kv_len = static_cast<int32_t>(s.kv_len);
    d.mask_base = s.mask_base;
    d.b = b;
    d.tiles = static_cast<int32_t>(tiles);
    d.heads = heads;
    d.descending = c1 >= c0 ? 1 : 0;
    entries.push_back(Entry{d, wmax});
  };
  // the query-side passes run one CTA per query head, the key-side pass one
  // per key/value head (it walks the query heads of its group)
  const int32_t nh = forward ? g.N : g.N_kv;
  if (g.layout == 0) {
    fill(plan.seqs[0], -1, static_cast<int32_t>(plan.B * nh));
  } else {
    for (int64_t b = 0; b < plan.B; ++b) fill(plan.seqs[b], static_cast<int32_t>(b), nh);
    std::stable_sort(entries.begin(), entries.end(),
                     [](const Entry& x, const Entry& y) { return x.weight > y.weight; });
  }
  std::vector<SeqDesc> out;
  out.reserve(entries.size());
  for (auto& e : entries) out.push_back(e.d);
  return out;
}

// Split the entries into launches of at most CAP entries and run `launch` on each table.
template <int CAP, typename F>
cudaError_t for_each_table(const std::vector<SeqDesc>& descs, size_t begin, size_t end, F&& launch) {
  static thread_local std::unique_ptr<SeqTable<CAP>> tab_storage;
  if (!tab_storage) tab_storage.reset(new SeqTable<CAP>());
  SeqTable<CAP>& tab = *tab_storage;
  for (size_t c = begin; c < end; c += CAP) {
    const size_t n = std::min<size_t>(CAP, end - c);
    std::memset(&tab, 0, sizeof tab);
    int64_t items = 0;
    for (size_t i = 0; i < n; ++i) {
      tab.d[i] = descs[c + i];
      tab.d[i].item_begin = static_cast<int32_t>(items);
      items += static_cast<int64_t>(descs[c + i].tiles) * descs[c + i].heads;
    }
    tab.count = static_cast<int32_t>(n);
    tab.n_items = static_cast<int32_t>(items);
    cudaError_t e = launch(tab);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <typename FS, typename FL>
cudaError_t run_tables(const std::vector<SeqDesc>& descs, FS&& small, FL&& large) {
  if (descs.empty()) return cudaSuccess;
  if (descs.size() <= static_cast<size_t>(kSmallTable))
    return for_each_table<kSmallTable>(descs, 0, descs.size(), small);
  return for_each_table<kLargeTable>(descs, 0, descs.size(), large);
}

// ------------------------------------------------------------ TMA maps --
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 128 rows x 64 columns per box, 128-byte swizzle.  BNSD: (d, s, n, b);
// TND: (d, n, t, 1).
swa_status_t make_map(CUtensorMap* m, const void* ptr, const Plan& plan, bool q_side, const char* name) {
  auto fn = encode_fn();
  if (!fn) return fail(SWA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const Geometry& g = plan.g;
  const cuuint64_t D = g.D, N = q_side ? g.N : g.N_kv;
  const cuuint64_t es_bytes = 2;
  const cuuint32_t box_x = 64;  // 128 bytes, one swizzle row
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4];
  const cuuint32_t es[4] = {1, 1, 1, 1};
  if (g.layout == 0) {
    const cuuint64_t S = q_side ? g.S_q : g.S_kv;
    dims[0] = D; dims[1] = S; dims[2] = N; dims[3] = static_cast<cuuint64_t>(plan.B);
    strides[0] = D * es_bytes; strides[1] = S * D * es_bytes; strides[2] = N * S * D * es_bytes;
    box[0] = box_x; box[1] = kTileM; box[2] = 1; box[3] = 1;
  } else {
    const cuuint64_t T = static_cast<cuuint64_t>(q_side ? plan.q_rows : plan.kv_rows);
    dims[0] = D; dims[1] = N; dims[2] = T; dims[3] = 1;
    strides[0] = D * es_bytes; strides[1] = N * D * es_bytes; strides[2] = T * N * D * es_bytes;
    box[0] = box_x; box[1] = 1; box[2] = kTileM; box[3] = 1;
  }
  CUresult r = fn(m, g.f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SWA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", name, (int)r);
  return SWA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

size_t q_elems(const Plan& plan) { return static_cast<size_t>(plan.q_rows) * plan.g.N * plan.g.D; }
size_t kv_elems(const Plan& plan) { return static_cast<size_t>(plan.kv_rows) * plan.g.N_kv * plan.g.D; }

// fp32 inputs: bf16 copies of q, k, v (and for the backward dy, out) follow
// the header / statistics in the workspace, each 256-byte aligned.
struct FwdLayout {
  size_t q16, k16, v16, total;
};
FwdLayout fwd_layout(const Plan& plan) {
  FwdLayout l{};
  l.total = kHeaderBytes;
  if (plan.g.out_f32) {
    l.q16 = l.total;
    l.k16 = l.q16 + round256(q_elems(plan) * 2);
    l.v16 = l.k16 + round256(kv_elems(plan) * 2);
    l.total = l.v16 + round256(kv_elems(plan) * 2);
  }
  return l;
}

struct BwdLayout {
  size_t lse2, dsum, q16, k16, v16, dy16, out16, total;
};
BwdLayout bwd_layout(const Plan& plan) {
  const size_t rows = static_cast<size_t>(plan.q_rows) * plan.g.N;
  BwdLayout l{};
  l.lse2 = kHeaderBytes;
  l.dsum = l.lse2 + round256(rows * 4);
  l.total = l.dsum + round256(rows * 4);
  if (plan.g.out_f32) {
    l.q16 = l.total;
    l.k16 = l.q16 + round256(q_elems(plan) * 2);
    l.v16 = l.k16 + round256(kv_elems(plan) * 2);
    l.dy16 = l.v16 + round256(kv_elems(plan) * 2);
    l.out16 = l.dy16 + round256(q_elems(plan) * 2);
    l.total = l.out16 + round256(q_elems(plan) * 2);
  }
  return l;
}

swa_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(SWA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

// Error text for entry points defined in other translation units.
swa_status_t swa::set_error(swa_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

// ------------------------------------------------------------------ ABI --
extern "C" {

void swa_params_default(swa_params_t* p) {
  if (!p) return;
  std::memset(p, 0, sizeof *p);
  p->scale = 1.0;
  p->keep_prob = 1.0;
  p->pre_tokens = 2147483647;
  p->next_tokens = 2147483647;
  p->sparse_mode = 0;
}

swa_status_t swa_forward_workspace_size(const swa_params_t* p, size_t* bytes) {
  if (!bytes) return fail(SWA_ERR_PARAM_NULLPTR, "bytes is NULL");
  Plan plan;
  swa_status_t st = make_plan(p, plan);
  if (st != SWA_OK) return st;
  *bytes = fwd_layout(plan).total;
  return SWA_OK;
}

swa_status_t swa_backward_workspace_size(const swa_params_t* p, size_t* bytes) {
  if (!bytes) return fail(SWA_ERR_PARAM_NULLPTR, "bytes is NULL");
  Plan plan;
  swa_status_t st = make_plan(p, plan);
  if (st != SWA_OK) return st;
  *bytes = bwd_layout(plan).total;
  return SWA_OK;
}

swa_status_t swa_forward(const swa_params_t* p, const void* q, const void* k, const void* v, const uint8_t* drop_mask,
                         void* out, float* softmax_max, float* softmax_sum, void* workspace, size_t workspace_bytes,
                         swa_stream_t stream) {
  Plan plan;
  swa_status_t st = make_plan(p, plan);
  if (st != SWA_OK) return st;
  if (!q || !k || !v || !out || !softmax_max || !softmax_sum)
    return fail(SWA_ERR_PARAM_NULLPTR, "a required tensor pointer is NULL");
  if ((p->keep_prob < 1.0 && p->dropout_gen == 0) != (drop_mask != nullptr))
    return fail(SWA_ERR_PARAM_INVALID,
                "drop_mask must be given iff keep_prob < 1 and dropout_gen == 0 (keep_prob = %g, dropout_gen = %d)",
                p->keep_prob, p->dropout_gen);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(softmax_max) ||
      !aligned16(softmax_sum) || !aligned16(drop_mask))
    return fail(SWA_ERR_PARAM_INVALID, "tensor pointers (and drop_mask) must be 16-byte aligned");
  const FwdLayout lay = fwd_layout(plan);
  if (!workspace || workspace_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(SWA_ERR_WORKSPACE, "workspace must be >= %zu bytes and 256-byte aligned (got %zu)", lay.total,
                workspace_bytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (plan.g.out_f32) {  // bf16 copies of the fp32 inputs
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const void* src[3] = {q, k, v};
    const size_t off[3] = {lay.q16, lay.k16, lay.v16}, n[3] = {q_elems(plan), kv_elems(plan), kv_elems(plan)};
    for (int t = 0; t < 3; ++t) {
      e = launch_to_bf16(static_cast<const float*>(src[t]), reinterpret_cast<__nv_bfloat16*>(ws + off[t]),
                         static_cast<int64_t>(n[t]), s);
      if (e != cudaSuccess) return cuda_fail(e, "fp32 -> bf16 conversion launch");
    }
    q = ws + lay.q16;
    k = ws + lay.k16;
    v = ws + lay.v16;
  }

  CUtensorMap mq, mk, mv;
  if ((st = make_map(&mq, q, plan, true, "q")) != SWA_OK) return st;
  if ((st = make_map(&mk, k, plan, false, "k")) != SWA_OK) return st;
  if ((st = make_map(&mv, v, plan, false, "v")) != SWA_OK) return st;

  FwdArgs a{};
  a.g = plan.g;
  a.mask = drop_mask;
  a.out = out;
  a.smax = softmax_max;
  a.ssum = softmax_sum;
  a.err = static_cast<int32_t*>(workspace);

  std::vector<SeqDesc> descs = build_descs(plan, true);
  if (descs.empty() || SWA_CHECKS) {  // otherwise the first launch clears the status word itself
    e = cudaMemsetAsync(workspace, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace header");
  }
  // D <= 64: TMEM holds two query tiles' S, O and P, and one CTA takes a pair
  // of consecutive query tiles (swa_fwd_pair.cu), when the pairs still fill
  // every SM at least once; smaller problems keep one CTA per query tile
  bool pair = false;
  if (plan.g.D <= 64) {
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "reading the SM count");
    int64_t items = 0;
    for (const SeqDesc& d : descs) items += static_cast<int64_t>(d.tiles) * d.heads;
    const int32_t mode = g_fwd_pairs.load(std::memory_order_relaxed);
    pair = mode == 1 || (mode == 0 && items >= 2 * static_cast<int64_t>(sms));
  }
  if (pair)
    for (SeqDesc& d : descs) d.tiles = (d.tiles + 1) / 2;
  if (t_ev[0]) cudaEventRecord(t_ev[0], s);
  int launches = 0;
  auto one = [&](const auto& t) {
    FwdArgs at = a;
    at.clear_err = (launches++ == 0 && !SWA_CHECKS) ? 1 : 0;
    return pair ? launch_forward_pair(at, t, mq, mk, mv, s) : launch_forward(at, t, mq, mk, mv, s);
  };
  e = run_tables(descs, one, one);
  if (t_ev[1]) cudaEventRecord(t_ev[1], s);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return SWA_OK;
}

swa_status_t swa_backward(const swa_params_t* p, const void* q, const void* k, const void* v, const void* dy,
                          const void* out, const float* softmax_max, const float* softmax_sum,
                          const uint8_t* drop_mask, void* dq, void* dk, void* dv, void* workspace,
                          size_t workspace_bytes, swa_stream_t stream) {
  Plan plan;
  swa_status_t st = make_plan(p, plan);
  if (st != SWA_OK) return st;
  if (!q || !k || !v || !dy || !out || !softmax_max || !softmax_sum || !dq || !dk || !dv)
    return fail(SWA_ERR_PARAM_NULLPTR, "a required tensor pointer is NULL");
  if ((p->keep_prob < 1.0 && p->dropout_gen == 0) != (drop_mask != nullptr))
    return fail(SWA_ERR_PARAM_INVALID,
                "drop_mask must be given iff keep_prob < 1 and dropout_gen == 0 (keep_prob = %g, dropout_gen = %d)",
                p->keep_prob, p->dropout_gen);
  for (const void* ptr : {q, k, v, dy, out, static_cast<const void*>(drop_mask), static_cast<const void*>(softmax_max),
                          static_cast<const void*>(softmax_sum), static_cast<const void*>(dq),
                          static_cast<const void*>(dk), static_cast<const void*>(dv)})
    if (!aligned16(ptr)) return fail(SWA_ERR_PARAM_INVALID, "tensor pointers must be 16-byte aligned");
  const BwdLayout lay = bwd_layout(plan);
  if (!workspace || workspace_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(SWA_ERR_WORKSPACE, "workspace must be >= %zu bytes and 256-byte aligned (got %zu)", lay.total,
                workspace_bytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (plan.g.out_f32) {  // bf16 copies of the fp32 inputs (out only feeds the preprocess)
    const void* src[5] = {q, k, v, dy, out};
    const size_t off[5] = {lay.q16, lay.k16, lay.v16, lay.dy16, lay.out16};
    const size_t n[5] = {q_elems(plan), kv_elems(plan), kv_elems(plan), q_elems(plan), q_elems(plan)};
    for (int t = 0; t < 5; ++t) {
      const cudaError_t ce = launch_to_bf16(static_cast<const float*>(src[t]),
                                            reinterpret_cast<__nv_bfloat16*>(ws + off[t]),
                                            static_cast<int64_t>(n[t]), s);
      if (ce != cudaSuccess) return cuda_fail(ce, "fp32 -> bf16 conversion launch");
    }
    q = ws + lay.q16;
    k = ws + lay.k16;
    v = ws + lay.v16;
    dy = ws + lay.dy16;
    out = ws + lay.out16;
  }

  CUtensorMap mq, mk, mv, mdy;
  if ((st = make_map(&mq, q, plan, true, "q")) != SWA_OK) return st;
  if ((st = make_map(&mk, k, plan, false, "k")) != SWA_OK) return st;
  if ((st = make_map(&mv, v, plan, false, "v")) != SWA_OK) return st;
  if ((st = make_map(&mdy, dy, plan, true, "dy")) != SWA_OK) return st;

  float* lse2 = reinterpret_cast<float*>(ws + lay.lse2);
  float* dsum = reinterpret_cast<float*>(ws + lay.dsum);
  const int64_t rows = plan.q_rows * plan.g.N;

  PrepArgs pa{};
  pa.g = plan.g;
  pa.rows = rows;
  pa.err = reinterpret_cast<int32_t*>(ws);
  pa.dy = static_cast<const __nv_bfloat16*>(dy);
  pa.out = static_cast<const __nv_bfloat16*>(out);
  pa.smax = softmax_max;
  pa.ssum = softmax_sum;
  pa.lse2 = lse2;
  pa.dsum = dsum;
  cudaError_t e = cudaSuccess;
  if (SWA_CHECKS) {  // the release preprocess clears the status word itself
    e = cudaMemsetAsync(ws, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace header");
  }
  if (t_ev[6]) cudaEventRecord(t_ev[6], s);
  e = launch_prep(pa, s);
  if (t_ev[7]) cudaEventRecord(t_ev[7], s);
  if (e != cudaSuccess) return cuda_fail(e, "backward preprocess launch");

  BwdArgs a{};
  a.g = plan.g;
  a.mask = drop_mask;
  a.lse2 = lse2;
  a.dsum = dsum;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.err = reinterpret_cast<int32_t*>(ws);
  // key-major pass: dK, dV (one work item per key tile)
  const std::vector<SeqDesc> kv_descs = build_descs(plan, false);
  if (t_ev[2]) cudaEventRecord(t_ev[2], s);
  e = run_tables(
      kv_descs, [&](const SeqTable<kSmallTable>& t) { return launch_backward_dkv(a, t, mq, mk, mv, mdy, s); },
      [&](const SeqTable<kLargeTable>& t) { return launch_backward_dkv(a, t, mq, mk, mv, mdy, s); });
  if (t_ev[3]) cudaEventRecord(t_ev[3], s);
  if (e != cudaSuccess) return cuda_fail(e, "backward dK/dV launch");
  // query-major pass: dQ (one work item per query tile)
  const std::vector<SeqDesc> q_descs = build_descs(plan, true);
  if (t_ev[4]) cudaEventRecord(t_ev[4], s);
  e = run_tables(
      q_descs, [&](const SeqTable<kSmallTable>& t) { return launch_backward_dq(a, t, mq, mk, mv, mdy, s); },
      [&](const SeqTable<kLargeTable>& t) { return launch_backward_dq(a, t, mq, mk, mv, mdy, s); });
  if (t_ev[5]) cudaEventRecord(t_ev[5], s);
  if (e != cudaSuccess) return cuda_fail(e, "backward dQ launch");
  return SWA_OK;
}

swa_status_t swa_dropout_mask(const swa_params_t* p, uint8_t* mask, size_t mask_bytes, swa_stream_t stream) {
  Plan plan;
  swa_status_t st = make_plan(p, plan);
  if (st != SWA_OK) return st;
  if (!mask) return fail(SWA_ERR_PARAM_NULLPTR, "mask is NULL");
  const size_t need = static_cast<size_t>((plan.mask_bits + 127) / 128) * 16;
  if (mask_bytes < need)
    return fail(SWA_ERR_WORKSPACE, "mask needs %zu bytes (16-byte multiple of the packed bits), got %zu", need,
                mask_bytes);
  if (!aligned16(mask)) return fail(SWA_ERR_PARAM_INVALID, "mask must be 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(mask, 0, mask_bytes, s);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the mask");
  MaskGenArgs a{};
  a.g = plan.g;
  a.mask = reinterpret_cast<uint32_t*>(mask);
  const std::vector<SeqDesc> descs = build_descs(plan, true);
  e = run_tables(
      descs, [&](const SeqTable<kSmallTable>& t) { return launch_dropout_mask(a, t, s); },
      [&](const SeqTable<kLargeTable>& t) { return launch_dropout_mask(a, t, s); });
  if (e != cudaSuccess) return cuda_fail(e, "dropout mask launch");
  return SWA_OK;
}

swa_status_t swa_workspace_status(const void* workspace, swa_stream_t stream) {
  if (!workspace) return fail(SWA_ERR_PARAM_NULLPTR, "workspace is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int32_t word = 0;
  e = cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the workspace header");
  if (word == kErrBounds)
    return fail(SWA_ERR_BOUNDS, "the bounds-checked build skipped an access outside its tensor (code %d)", word);
  if (word != 0) return fail(SWA_ERR_TIMEOUT, "a kernel gave up a bounded wait (code %d)", word);
  return SWA_OK;
}

swa_status_t swa_debug_schedule(const swa_params_t* p, int32_t pass, int32_t* items, int64_t capacity,
                                int64_t* count) {
  if (!count) return fail(SWA_ERR_PARAM_NULLPTR, "count is NULL");
  if (pass < 0 || pass > 2) return fail(SWA_ERR_PARAM_INVALID, "pass should be 0, 1 or 2, got %d", pass);
  Plan plan;
  swa_status_t st = make_plan(p, plan);
  if (st != SWA_OK) return st;
  const bool query_side = pass != 1;
  const int nh = query_side ? plan.g.N : plan.g.N_kv;
  std::vector<SeqDesc> descs = build_descs(plan, query_side);
  if (pass == 2)  // the forward's pairs of query tiles (as swa_forward sets them up at D <= 64)
    for (SeqDesc& d : descs) d.tiles = (d.tiles + 1) / 2;
  int64_t n = 0;
  int32_t launch = 0;
  auto emit = [&](const auto& tab) -> cudaError_t {
    for (int k = 0; k < tab.n_items; ++k) {
      const Item it = resolve_item(tab, plan.g, k, nh);
      int t0, cnt;
      if (pass == 0) key_tiles_of_query_tile(plan.g, it.s, it.tile, &t0, &cnt);
      else if (pass == 1) query_tiles_of_key_tile(plan.g, it.s, it.tile, &t0, &cnt);
      else key_tiles_of_query_pair(plan.g, it.s, it.tile, &t0, &cnt);
      if (items && n < capacity) {
        int32_t* r = items + 6 * n;
        r[0] = launch;
        r[1] = it.b;
        r[2] = it.n;
        r[3] = it.tile;
        r[4] = t0;
        r[5] = cnt;
      }
      ++n;
    }
    ++launch;
    return cudaSuccess;
  };
  run_tables(descs, emit, emit);
  *count = n;
  return SWA_OK;
}

void swa_debug_stall(int32_t kernels) { g_stall.store(kernels & 7, std::memory_order_relaxed); }
void swa_debug_extent_slack(int64_t elems) { g_extent_slack.store(std::max<int64_t>(elems, 0), std::memory_order_relaxed); }
void swa_debug_forward_pairs(int32_t mode) {
  g_fwd_pairs.store(mode >= 0 && mode <= 2 ? mode : 0, std::memory_order_relaxed);
}

void swa_set_timing_events(void* const* events) {
  for (int i = 0; i < 8; ++i) t_ev[i] = events ? static_cast<cudaEvent_t>(events[i]) : nullptr;
}

const char* swa_last_error(void) { return t_last_error.c_str(); }

}  // extern "C"
