// swa_host.cpp — swa_step_host: forward + backward of a problem whose inputs
// and outputs live in host memory, with the host <-> device copies overlapped
// with the computation.
//
// The heads are split into `chunks` equal groups (the first and the last
// split further into halves, see StepPlan).  Each group is a complete
// smaller problem (heads are independent in every step of the method), so it
// is copied into its own compact device tensors, computed by swa_forward and
// swa_backward, and copied back.  Chunk c+1's inputs travel host -> device on
// one stream and chunk c-1's results device -> host on others while chunk c
// computes.  Consecutive chunks compute on two internal streams in turn, so
// the kernels of chunk c+1 can start on the SMs that chunk c's last wave of
// CTAs leaves idle: smaller chunks (a shorter pipeline fill and drain of the
// copies) then cost no kernel efficiency.  Each compute stream has its own
// device -> host stream: a chunk's results queue behind its own backward,
// not behind the other stream's chunk, so the device -> host direction of
// the link (the one that drains last) is not left idle while a ready chunk
// waits.  A head group of a BNSD tensor is
// one contiguous block per batch, and of a TND tensor one block per row, so
// every copy is a single 2-D copy (rows = batches or tokens, pitch = the full
// row).
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "swa.h"
#include "swa_internal.h"

namespace {

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// ------------------------------------------------ streams and events --
// The internal streams and events of swa_step_host are created once per CUDA
// context and kept for the life of the process.  Creating and destroying five
// streams and some seventy events on every call took 0.5 ms of host time, and
// now and then a call stalled ~9 ms inside those driver calls (measured on
// BNSD 1x32x32768x128 in 16 head groups: one step in a dozen took 16 ms
// instead of 7.6), delaying the whole step.  A context is told apart by its unique id (cuCtxGetId), so
// that a context created after cudaDeviceReset gets a set of its own and
// never touches handles of the destroyed one.  A call holds g_step_mu while
// it enqueues: another call cannot re-record one of its events before the
// waits on it are queued.  (Re-recording an event whose earlier record is
// still pending on the GPU is fine: a wait is bound to the record that
// preceded it.)
struct StepStreams {
  unsigned long long ctx = 0;
  cudaStream_t s_in = nullptr, s_outs[2] = {nullptr, nullptr}, s_comp[2] = {nullptr, nullptr};
  std::vector<cudaEvent_t> events;
};
std::mutex g_step_mu;
std::vector<StepStreams*> g_step_sets;  // guarded by g_step_mu; kept until the process exits

// Unique id of the context current on this thread: the caller's own context
// if it made one current, else the runtime's primary context of the current
// device, which the runtime makes current on its first use in the thread.
cudaError_t current_context_id(unsigned long long* id) {
  static std::once_flag once;
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  if (!get_current || !get_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (!ctx) {  // no context current yet: a no-op runtime call binds the primary one
    const cudaError_t e = cudaFree(nullptr);
    if (e != cudaSuccess) return e;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
  }
  if (get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}

// The set of the current context, created on first use.  Call with g_step_mu held.
cudaError_t step_streams(StepStreams** out) {
  unsigned long long id = 0;
  cudaError_t e = current_context_id(&id);
  if (e != cudaSuccess) return e;
  for (StepStreams* x : g_step_sets)
    if (x->ctx == id) {
      *out = x;
      return cudaSuccess;
    }
  StepStreams* x = new StepStreams;
  x->ctx = id;
  e = cudaStreamCreateWithFlags(&x->s_in, cudaStreamNonBlocking);
  for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamCreateWithFlags(&x->s_outs[i], cudaStreamNonBlocking);
  for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamCreateWithFlags(&x->s_comp[i], cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    for (cudaStream_t st : {x->s_in, x->s_outs[0], x->s_outs[1], x->s_comp[0], x->s_comp[1]})
      if (st) cudaStreamDestroy(st);
    delete x;
    return e;
  }
  g_step_sets.push_back(x);
  *out = x;
  return cudaSuccess;
}

// Copy geometry of one tensor for one head group: `rows` rows of `width`
// bytes at `pitch` on the host, packed back to back on the device.
struct Span {
  size_t rows = 0, width = 0, pitch = 0, first = 0;  // first: byte offset of head group 0's first row
  size_t dev_bytes() const { return rows * width; }
  size_t host_offset(int c) const { return first + static_cast<size_t>(c) * width; }
};

struct Layout {
  swa_params_t sub;             // the per-chunk problem
  Span q, kv, st;               // q-like (q, dy, out, dq), k-like (k, v, dk, dv), statistics
  size_t q_off, k_off, v_off, dy_off, out_off, dq_off, dk_off, dv_off, smax_off, ssum_off;  // within a chunk
  size_t fws_off, bws_off, chunk_bytes;
  size_t fws_bytes, bws_bytes;
  size_t total;
};

swa_status_t make_layout(const swa_params_t* p, int chunks, Layout& L) {
  if (!p) return swa::set_error(SWA_ERR_PARAM_NULLPTR, "params is NULL");
  if (chunks < 1) return swa::set_error(SWA_ERR_PARAM_INVALID, "chunks must be >= 1, got %d", chunks);
  const int64_t n_kv = p->N_kv == 0 ? p->N : p->N_kv;
  if (p->N % chunks != 0 || n_kv % chunks != 0)
    return swa::set_error(SWA_ERR_PARAM_INVALID, "chunks = %d must divide N = %lld and N_kv = %lld", chunks,
                          (long long)p->N, (long long)n_kv);
  if (p->keep_prob < 1.0 && (p->dropout_gen == 0 || chunks != 1))
    return swa::set_error(SWA_ERR_PARAM_INVALID,
                          "swa_step_host takes no drop_mask: dropout needs dropout_gen = 1 and chunks = 1 "
                          "(the generated keep bits are indexed by the whole problem's heads)");
  L.sub = *p;
  L.sub.N = p->N / chunks;
  L.sub.N_kv = p->N_kv == 0 ? 0 : p->N_kv / chunks;
  // validates everything else, on the chunk's problem
  swa_status_t st = swa_forward_workspace_size(&L.sub, &L.fws_bytes);
  if (st != SWA_OK) return st;
  if ((st = swa_backward_workspace_size(&L.sub, &L.bws_bytes)) != SWA_OK) return st;

  const size_t elt = p->dtype == SWA_DTYPE_FP32 ? 4 : 2;
  const size_t D = static_cast<size_t>(p->D), Nq = static_cast<size_t>(p->N), Nk = static_cast<size_t>(n_kv);
  const size_t nq = Nq / chunks, nk = Nk / chunks;
  if (p->layout == SWA_LAYOUT_BNSD) {
    const size_t B = static_cast<size_t>(p->B), Sq = static_cast<size_t>(p->S_q), Sk = static_cast<size_t>(p->S_kv);
    L.q = Span{B, nq * Sq * D * elt, Nq * Sq * D * elt, 0};
    L.kv = Span{B, nk * Sk * D * elt, Nk * Sk * D * elt, 0};
    L.st = Span{B, nq * Sq * 4, Nq * Sq * 4, 0};
  } else {
    const size_t Tq = static_cast<size_t>(p->T_q), Tk = static_cast<size_t>(p->T_kv);
    L.q = Span{Tq, nq * D * elt, Nq * D * elt, 0};
    L.kv = Span{Tk, nk * D * elt, Nk * D * elt, 0};
    L.st = Span{Tq, nq * 4, Nq * 4, 0};
  }
  size_t o = 0;
  auto take = [&o](size_t bytes) { const size_t at = o; o += round256(bytes); return at; };
  L.q_off = take(L.q.dev_bytes());
  L.k_off = take(L.kv.dev_bytes());
  L.v_off = take(L.kv.dev_bytes());
  L.dy_off = take(L.q.dev_bytes());
  L.out_off = take(L.q.dev_bytes());
  L.dq_off = take(L.q.dev_bytes());
  L.dk_off = take(L.kv.dev_bytes());
  L.dv_off = take(L.kv.dev_bytes());
  L.smax_off = take(L.st.dev_bytes());
  L.ssum_off = take(L.st.dev_bytes());
  L.fws_off = take(L.fws_bytes);  // each chunk keeps its own status words
  L.bws_off = take(L.bws_bytes);
  L.chunk_bytes = o;
  L.total = o * static_cast<size_t>(chunks);
  return SWA_OK;
}

// The pipeline's units: head groups of N / chunks heads, except at the two
// ends.  The first group is split in halves, its first half again, and so on
// for `levels` levels (while 2^levels * chunks divides N and N_kv, at most 3),
// and the last group the same way mirrored: with 8 groups of 4 heads the units
// hold 1, 1, 2, 4, ..., 4, 2, 1, 1 heads.  The pipeline's fill (the first
// unit's inputs) and drain (the last unit's results) then move a fraction of
// a group's bytes while the middle groups stay large.  Units are packed back
// to back in the device buffer.
struct Unit {
  const Layout* L;
  int group;   // head group index within L's split
  size_t off;  // byte offset of the unit's region in the device buffer
};
constexpr int kMaxLevels = 3;
struct StepPlan {
  Layout split[kMaxLevels + 1];  // split[l]: chunks * 2^l equal groups
  std::vector<Unit> units;
  size_t total = 0;
};

swa_status_t make_step_plan(const swa_params_t* p, int chunks, StepPlan& P) {
  swa_status_t st = make_layout(p, chunks, P.split[0]);
  if (st != SWA_OK) return st;
  const int64_t n_kv = p->N_kv == 0 ? p->N : p->N_kv;
  int levels = 0;
  while (chunks >= 2 && levels < kMaxLevels) {
    const int64_t g = int64_t{chunks} << (levels + 1);
    if (p->N % g != 0 || n_kv % g != 0) break;
    if ((st = make_layout(p, static_cast<int>(g), P.split[levels + 1])) != SWA_OK) return st;
    ++levels;
  }
  P.units.clear();
  size_t o = 0;
  auto add = [&](int l, int group) {
    P.units.push_back(Unit{&P.split[l], group, o});
    o += P.split[l].chunk_bytes;
  };
  if (levels == 0) {
    for (int c = 0; c < chunks; ++c) add(0, c);
  } else {
    // first group: split[levels] groups 0 and 1, then group 1 of each coarser split
    add(levels, 0);
    for (int l = levels; l >= 1; --l) add(l, 1);
    for (int c = 1; c < chunks - 1; ++c) add(0, c);
    // last group, mirrored: group 2^l * chunks - 2 of each finer split, then the last one
    for (int l = 1; l <= levels; ++l) add(l, (chunks << l) - 2);
    add(levels, (chunks << levels) - 1);
  }
  P.total = o;
  return SWA_OK;
}

cudaError_t copy_in(const Span& s, int c, void* dev, const void* host, cudaStream_t st) {
  return cudaMemcpy2DAsync(dev, s.width, static_cast<const uint8_t*>(host) + s.host_offset(c), s.pitch, s.width,
                           s.rows, cudaMemcpyHostToDevice, st);
}
cudaError_t copy_out(const Span& s, int c, void* host, const void* dev, cudaStream_t st) {
  return cudaMemcpy2DAsync(static_cast<uint8_t*>(host) + s.host_offset(c), s.pitch, dev, s.width, s.width, s.rows,
                           cudaMemcpyDeviceToHost, st);
}

swa_status_t cuda_fail(cudaError_t e, const char* what) {
  return swa::set_error(SWA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

extern "C" {

swa_status_t swa_step_host_buffer_size(const swa_params_t* p, int chunks, size_t* bytes) {
  if (!bytes) return swa::set_error(SWA_ERR_PARAM_NULLPTR, "bytes is NULL");
  StepPlan P;
  swa_status_t st = make_step_plan(p, chunks, P);
  if (st != SWA_OK) return st;
  *bytes = P.total;
  return SWA_OK;
}

swa_status_t swa_step_host(const swa_params_t* p, int chunks, const void* q, const void* k, const void* v,
                           const void* dy, void* out, float* softmax_max, float* softmax_sum, void* dq, void* dk,
                           void* dv, void* device_buffer, size_t device_bytes, swa_stream_t stream) {
  StepPlan P;
  swa_status_t st = make_step_plan(p, chunks, P);
  if (st != SWA_OK) return st;
  if (!q || !k || !v || !dy || !out || !softmax_max || !softmax_sum || !dq || !dk || !dv)
    return swa::set_error(SWA_ERR_PARAM_NULLPTR, "a required host pointer is NULL");
  if (!device_buffer || device_bytes < P.total || (reinterpret_cast<uintptr_t>(device_buffer) & 255u))
    return swa::set_error(SWA_ERR_WORKSPACE, "device_buffer must be >= %zu bytes and 256-byte aligned (got %zu)",
                          P.total, device_bytes);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // One host -> device stream, two compute streams with a device -> host
  // stream each, and events from the context's pool (StepStreams).
  std::lock_guard<std::mutex> lock(g_step_mu);
  StepStreams* set = nullptr;
  cudaError_t e = step_streams(&set);
  if (e != cudaSuccess) return cuda_fail(e, "setting up the copy streams");
  cudaStream_t s_in = set->s_in, s_outs[2] = {set->s_outs[0], set->s_outs[1]},
               s_comp[2] = {set->s_comp[0], set->s_comp[1]};
  size_t n_ev = 0;  // events of the pool taken by this call
  auto event = [&](cudaEvent_t* ev) {
    if (n_ev == set->events.size()) {
      cudaEvent_t fresh = nullptr;
      const cudaError_t r = cudaEventCreateWithFlags(&fresh, cudaEventDisableTiming);
      if (r != cudaSuccess) return r;
      set->events.push_back(fresh);
    }
    *ev = set->events[n_ev++];
    return cudaSuccess;
  };
  cudaEvent_t start = nullptr, done = nullptr;
  if (e == cudaSuccess) e = event(&start);
  if (e == cudaSuccess) e = event(&done);
  // nothing may start before what the caller queued earlier (which may still use the buffer)
  if (e == cudaSuccess) e = cudaEventRecord(start, cs);
  for (cudaStream_t x : {s_in, s_outs[0], s_outs[1], s_comp[0], s_comp[1]})
    if (e == cudaSuccess) e = cudaStreamWaitEvent(x, start, 0);
  if (e != cudaSuccess) return cuda_fail(e, "setting up the copy streams");
  uint8_t* base = static_cast<uint8_t*>(device_buffer);
  for (size_t u = 0; u < P.units.size(); ++u) {
    const Layout& L = *P.units[u].L;
    const int c = P.units[u].group;
    uint8_t* d = base + P.units[u].off;
    cudaStream_t comp = s_comp[u & 1], s_out = s_outs[u & 1];
    const swa_stream_t comp_h = reinterpret_cast<swa_stream_t>(comp);
    // The forward needs q, k, v only: it starts while dy is still being
    // copied.  out and the statistics are final after the forward and go
    // back while the backward runs.  (This shortens the pipeline's fill by
    // the first chunk's dy and its drain by the last chunk's out.)
    cudaEvent_t qkv_done = nullptr, dy_done = nullptr, fwd_done = nullptr, comp_done = nullptr;
    if ((e = event(&qkv_done)) != cudaSuccess || (e = event(&dy_done)) != cudaSuccess ||
        (e = event(&fwd_done)) != cudaSuccess || (e = event(&comp_done)) != cudaSuccess)
      break;
    if ((e = copy_in(L.q, c, d + L.q_off, q, s_in)) != cudaSuccess) break;
    if ((e = copy_in(L.kv, c, d + L.k_off, k, s_in)) != cudaSuccess) break;
    if ((e = copy_in(L.kv, c, d + L.v_off, v, s_in)) != cudaSuccess) break;
    if ((e = cudaEventRecord(qkv_done, s_in)) != cudaSuccess) break;
    if ((e = copy_in(L.q, c, d + L.dy_off, dy, s_in)) != cudaSuccess) break;
    if ((e = cudaEventRecord(dy_done, s_in)) != cudaSuccess) break;
    if ((e = cudaStreamWaitEvent(comp, qkv_done, 0)) != cudaSuccess) break;
    st = swa_forward(&L.sub, d + L.q_off, d + L.k_off, d + L.v_off, nullptr, d + L.out_off,
                     reinterpret_cast<float*>(d + L.smax_off), reinterpret_cast<float*>(d + L.ssum_off),
                     d + L.fws_off, L.fws_bytes, comp_h);
    if (st != SWA_OK) break;
    if ((e = cudaEventRecord(fwd_done, comp)) != cudaSuccess) break;
    if ((e = cudaStreamWaitEvent(s_out, fwd_done, 0)) != cudaSuccess) break;
    if ((e = copy_out(L.q, c, out, d + L.out_off, s_out)) != cudaSuccess) break;
    if ((e = copy_out(L.st, c, softmax_max, d + L.smax_off, s_out)) != cudaSuccess) break;
    if ((e = copy_out(L.st, c, softmax_sum, d + L.ssum_off, s_out)) != cudaSuccess) break;
    if ((e = cudaStreamWaitEvent(comp, dy_done, 0)) != cudaSuccess) break;
    st = swa_backward(&L.sub, d + L.q_off, d + L.k_off, d + L.v_off, d + L.dy_off, d + L.out_off,
                      reinterpret_cast<const float*>(d + L.smax_off), reinterpret_cast<const float*>(d + L.ssum_off),
                      nullptr, d + L.dq_off, d + L.dk_off, d + L.dv_off, d + L.bws_off, L.bws_bytes, comp_h);
    if (st != SWA_OK) break;
    if ((e = cudaEventRecord(comp_done, comp)) != cudaSuccess) break;
    if ((e = cudaStreamWaitEvent(s_out, comp_done, 0)) != cudaSuccess) break;
    if ((e = copy_out(L.q, c, dq, d + L.dq_off, s_out)) != cudaSuccess) break;
    if ((e = copy_out(L.kv, c, dk, d + L.dk_off, s_out)) != cudaSuccess) break;
    if ((e = copy_out(L.kv, c, dv, d + L.dv_off, s_out)) != cudaSuccess) break;
  }
  // The caller's stream completes only after the last result has reached the
  // host, and, after a failure part-way, only after every copy already
  // enqueued on any copy stream has run: host memory is never written
  // once the caller has seen the stream finish.
  cudaEvent_t in_end = nullptr, comp_end[2] = {nullptr, nullptr};
  cudaError_t e_end = event(&in_end);
  if (e_end == cudaSuccess) e_end = cudaEventRecord(in_end, s_in);
  if (e_end == cudaSuccess) e_end = cudaStreamWaitEvent(cs, in_end, 0);
  for (int i = 0; i < 2; ++i) {
    if (e_end == cudaSuccess) e_end = event(&comp_end[i]);
    if (e_end == cudaSuccess) e_end = cudaEventRecord(comp_end[i], s_comp[i]);
    if (e_end == cudaSuccess) e_end = cudaStreamWaitEvent(cs, comp_end[i], 0);
  }
  cudaEvent_t done2 = nullptr;
  if (e_end == cudaSuccess) e_end = event(&done2);
  if (e_end == cudaSuccess) e_end = cudaEventRecord(done, s_outs[0]);
  if (e_end == cudaSuccess) e_end = cudaStreamWaitEvent(cs, done, 0);
  if (e_end == cudaSuccess) e_end = cudaEventRecord(done2, s_outs[1]);
  if (e_end == cudaSuccess) e_end = cudaStreamWaitEvent(cs, done2, 0);
  if (e == cudaSuccess) e = e_end;
  if (st != SWA_OK) return st;
  if (e != cudaSuccess) return cuda_fail(e, "host step copies");
  return SWA_OK;
}

swa_status_t swa_step_host_status(const swa_params_t* p, int chunks, const void* device_buffer,
                                  swa_stream_t stream) {
  StepPlan P;
  swa_status_t st = make_step_plan(p, chunks, P);
  if (st != SWA_OK) return st;
  if (!device_buffer) return swa::set_error(SWA_ERR_PARAM_NULLPTR, "device_buffer is NULL");
  const uint8_t* base = static_cast<const uint8_t*>(device_buffer);
  for (const Unit& un : P.units) {
    const uint8_t* d = base + un.off;
    if ((st = swa_workspace_status(d + un.L->fws_off, stream)) != SWA_OK) return st;
    if ((st = swa_workspace_status(d + un.L->bws_off, stream)) != SWA_OK) return st;
  }
  return SWA_OK;
}

}  // extern "C"
