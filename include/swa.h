/*
 * swa.h — C ABI of libswa: sliding-window (BAND) / unmasked FlashAttention
 * forward and backward on GB300 (sm_103a).
 *
 * The operation (FlashAttentionVarLenScore doc, "计算公式"; PyPTO-Gym
 * FlashAttentionScoreGrad article, "前向公式" / "反向公式"):
 *
 *   forward   O = Dropout(Softmax(Mask(scale * Q K^T)), keep_prob) V
 *             softmax_max_i = max_{j visible} scale * q_i.k_j
 *             softmax_sum_i = sum_{j visible} exp(scale * q_i.k_j - softmax_max_i)
 *   backward  P  = exp(scale * Q K^T - softmax_max) / softmax_sum
 *             D  = rowsum(dY * O)
 *             dP = (dY V^T) * z / keep_prob
 *             dS = P * (dP - D)
 *             dV = (P * z / keep_prob)^T dY,  dQ = scale dS K,  dK = scale dS^T Q
 *
 * Mask ("sparse_mode", FlashAttentionVarLenScore doc, parameter
 * sparseModeOptional; the split into swa_forward / swa_backward limited to
 * modes 0 and 4 follows the pzsr.cn article, §1.2 and §3):
 *   0  no mask: query i sees every key of its sequence;
 *   4  BAND: query i sees key j iff  i - pre_tokens <= j <= i + next_tokens
 *      (indices local to the sequence, top-left aligned when Sq != Skv).
 * A query row that sees no key gets out = 0, softmax_max = -inf,
 * softmax_sum = 0 and a zero dq row; it contributes nothing to dk / dv.
 *
 * Dropout (doc parameter dropMaskOptional / keepProbOptional): drop_mask is
 * a packed bit mask, 8 elements per byte, least significant bit first,
 * 1 = keep.  Element order: BNSD e = ((b*N + n)*Sq + i)*Skv + j; TND
 * e = sum_{b'<b} N*Sq_b'*Skv_b' + (n*Sq_b + i)*Skv_b + j (no padding).
 * softmax_sum excludes dropout; kept probabilities are scaled by 1/keep_prob.
 * Instead of a mask, a seed and an offset may stand for it (dropout_gen = 1;
 * the pages' high-level backward regenerates the mask from seed / offset,
 * SWA article §1.1): element (query row r, local key j) is kept iff byte
 * (j mod 16) of Philox4x32-10(counter = (j/16, lo32 r, hi32 r,
 * lo32 dropout_offset), key = (lo32 dropout_seed, hi32 dropout_seed)),
 * bytes little-endian across the four output words, is below
 * round(keep_prob * 256); r is the statistics index of the row (BNSD
 * (b*N + n)*S_q + i, TND t*N + n).  swa_dropout_mask writes that mask out.
 *
 * Layouts (doc parameter list, inputLayout; PyPTO-Gym article, I/O table):
 *   BNSD  q, dy, out, dq: [B, N, S_q, D];  k, v, dk, dv: [B, N, S_kv, D]
 *         softmax_max / softmax_sum: [B, N, S_q] fp32
 *   TND   q, dy, out, dq: [T_q, N, D];     k, v, dk, dv: [T_kv, N, D]
 *         softmax_max / softmax_sum: [T_q, N] fp32
 *   All tensors are dense, row-major, of p->dtype (bf16 by default) unless
 *   stated (statistics are fp32), device memory,
 *   16-byte aligned.  D is a multiple of 8 from 8 to 128 (a row of D
 *   elements then starts on a 16-byte boundary).  The kernels compute on 64
 *   (D <= 64) or 128 columns per row; the tensor maps fill the columns past D
 *   with zeros, which changes no result, and nothing past D is written.  The
 *   grad API's own pre-processing pads special head dims such as 72 and 88
 *   (aclnnFlashAttentionUnpaddingScoreGradV2 article §8.2, the API layer);
 *   here the padding costs no copy.
 *
 * Variable length (TND): cu_seqlens_q / cu_seqlens_kv are HOST arrays of
 * length B holding cumulative sequence ends without a leading 0 (doc
 * parameters actualSeqQLenOptional / actualSeqKvLenOptional).  A length-0
 * sequence is allowed; a trailing run of zeros marks skipped batches
 * (aclnnFlashAttentionUnpaddingScoreGradV2 article, §6.4).  The last
 * non-zero entry must equal T.
 *
 * Two-phase calls (doc, "两段式接口"): ask for the workspace size, let the
 * caller allocate it in device memory, then call.  The library allocates
 * nothing, keeps no pointer after a call returns and reads host arrays only
 * during the call.  Calls only enqueue work on `stream` (a cudaStream_t) and
 * return; results are ready when the stream is.  A workspace may be reused
 * by later calls on the same stream but not by calls running concurrently.
 *
 * Status codes follow the aclnn numbering (doc, "返回值").
 */
#ifndef SWA_H
#define SWA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SWA_API __attribute__((visibility("default")))
#else
#define SWA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *swa_stream_t; /* same type as cudaStream_t */

typedef enum { SWA_LAYOUT_BNSD = 0, SWA_LAYOUT_TND = 1 } swa_layout_t;

typedef enum {
  SWA_OK = 0,
  SWA_ERR_PARAM_NULLPTR = 161001, /* a required pointer is NULL */
  SWA_ERR_PARAM_INVALID = 161002, /* a value is outside its documented range */
  SWA_ERR_UNSUPPORTED = 161100,   /* valid per the API but not built (e.g. D past 128 or not a multiple of 8) */
  SWA_ERR_WORKSPACE = 161101,     /* workspace NULL or smaller than the size query says */
  SWA_ERR_CUDA = 161102,          /* a CUDA runtime call failed (text in swa_last_error) */
  SWA_ERR_TIMEOUT = 161103,       /* a kernel gave up a bounded wait (swa_workspace_status) */
  SWA_ERR_BOUNDS = 161104         /* bounds-checked build only: a kernel skipped an access outside its
                                     tensor (swa_workspace_status) */
} swa_status_t;

typedef struct {
  int32_t layout;               /* swa_layout_t */
  int64_t B, N, D;              /* batch, heads (headNum), head dim (8..128, a multiple of 8) */
  int64_t S_q, S_kv;            /* BNSD sequence lengths (ignored for TND) */
  int64_t T_q, T_kv;            /* TND total rows (ignored for BNSD) */
  const int64_t *cu_seqlens_q;  /* TND: host, length B, cumulative ends (see above) */
  const int64_t *cu_seqlens_kv; /* TND: host, length B */
  double scale;                 /* score scale, default 1.0, usually D^-0.5 */
  int64_t pre_tokens;           /* BAND left extent, default 2147483647 */
  int64_t next_tokens;          /* BAND right extent, default 2147483647 */
  int32_t sparse_mode;          /* 0 or 4 */
  double keep_prob;             /* dropout keep probability in (0, 1], default 1.0 */
  int64_t N_kv;                 /* key/value heads for grouped-query attention: N must be a
                                   multiple of N_kv (aclnnFlashAttentionUnpaddingScoreGradV2
                                   article, shape constraints: Nq/Nkv a non-zero integer);
                                   query head n reads key/value head n / (N / N_kv).
                                   k, v, dk, dv then have N_kv heads ([B,N_kv,S_kv,D] or
                                   [T_kv,N_kv,D]).  0 (the default) means N_kv = N. */
  int32_t dropout_gen;          /* 1: keep_prob < 1 with drop_mask NULL, the mask being the one
                                   dropout_seed / dropout_offset stand for (see above); 0: the
                                   caller's drop_mask.  Default 0. */
  uint64_t dropout_seed;
  uint64_t dropout_offset;
  int32_t dtype;                /* element type of q, k, v, dy, out, dq, dk, dv (doc: FLOAT16 /
                                   BFLOAT16 / FLOAT32): SWA_DTYPE_BF16 (0, default),
                                   SWA_DTYPE_FP16 (1) or SWA_DTYPE_FP32 (2).  fp32: the
                                   tensor-core operands are bf16 copies of the inputs
                                   (rounded to nearest even, made in the workspace), every
                                   accumulation is fp32 as for the other types, and the
                                   outputs are stored in fp32 */
} swa_params_t;

typedef enum { SWA_DTYPE_BF16 = 0, SWA_DTYPE_FP16 = 1, SWA_DTYPE_FP32 = 2 } swa_dtype_t;

/* Fill `p` with the documented defaults (FlashAttentionScore REG_OP
 * attribute defaults): scale 1.0, keep_prob 1.0, pre/next 2147483647,
 * sparse_mode 0; everything else zero / NULL. */
SWA_API void swa_params_default(swa_params_t *p);

/* Device workspace bytes that swa_forward needs for these parameters (a
 * status word; the work schedule travels as a kernel parameter; with fp32
 * inputs also bf16 copies of q, k and v).  Errors: SWA_ERR_PARAM_NULLPTR,
 * SWA_ERR_PARAM_INVALID, SWA_ERR_UNSUPPORTED. */
SWA_API swa_status_t swa_forward_workspace_size(const swa_params_t *p, size_t *bytes);

/* Forward (doc formula; PyPTO-Gym "前向公式").
 *   q, k, v       device, p->dtype (bf16 / fp16 / fp32), layout per p->layout
 *   drop_mask     device, packed keep bits, 16-byte aligned; NULL iff keep_prob == 1
 *                 or dropout_gen == 1
 *   out           device, p->dtype, q's shape
 *   softmax_max   device, fp32, [B,N,S_q] or [T_q,N]
 *   softmax_sum   device, fp32, same shape
 *   workspace     device, >= swa_forward_workspace_size bytes, 256-byte aligned
 * Errors: the size query's, plus SWA_ERR_WORKSPACE and SWA_ERR_CUDA.  Nothing
 * is enqueued when a status other than SWA_OK is returned. */
SWA_API swa_status_t swa_forward(const swa_params_t *p, const void *q, const void *k, const void *v,
                         const uint8_t *drop_mask, void *out, float *softmax_max, float *softmax_sum,
                         void *workspace, size_t workspace_bytes, swa_stream_t stream);

/* Device workspace bytes that swa_backward needs: a status word, and per
 * query row D = rowsum(dY*O) and the log2-sum-exp of the forward statistics
 * (8 bytes per query row and head); with fp32 inputs also bf16 copies of q,
 * k, v, dy and out. */
SWA_API swa_status_t swa_backward_workspace_size(const swa_params_t *p, size_t *bytes);

/* Backward (PyPTO-Gym "反向公式"; aclnnFlashAttentionUnpaddingScoreGradV2
 * article §2.3).  out / softmax_max / softmax_sum are this library's forward
 * results for the same q, k, v, drop_mask and parameters.
 *   dy            device, p->dtype, q's shape (gradient of out)
 *   dq, dk, dv    device, p->dtype, shapes of q, k, v; fully overwritten
 * Errors: as swa_forward. */
SWA_API swa_status_t swa_backward(const swa_params_t *p, const void *q, const void *k, const void *v, const void *dy,
                          const void *out, const float *softmax_max, const float *softmax_sum,
                          const uint8_t *drop_mask, void *dq, void *dk, void *dv, void *workspace,
                          size_t workspace_bytes, swa_stream_t stream);

/* swa_backward without a workspace argument, for callers that cannot hand the
 * library device memory (the pages have no counterpart; this is an addition of
 * this library).  Example callers: a plugin inside a framework that owns all
 * device memory through its own pool and forbids extra cudaMalloc calls, or a
 * latency-critical loop that must not allocate after start-up.
 *
 * Arguments and results are those of swa_backward.  The scratch it needs
 * (status word, per-row D and log2-sum-exp) lives in a
 * fixed 64 MiB device array compiled into the library: every GPU that loads
 * the library keeps it until the process exits.  A problem needing more than
 * 64 MiB of scratch (swa_backward_workspace_size) is rejected with
 * SWA_ERR_WORKSPACE.  Every call looks up the array's device address in the
 * current context (cudaGetSymbolAddress), so an address never outlives its
 * context; the first lookup on a device may load the library's device code,
 * so make the first call before any stream capture.  The library carries its
 * own copy of the CUDA runtime (linked statically): do not reset the device
 * (cudaDeviceReset, or a primary-context reset through the driver) between
 * calls while the library stays loaded, since whether its runtime then
 * reloads its device code is not specified.  All calls on a device
 * share the array and
 * each call clears what must start at zero, so calls whose kernels overlap on
 * the GPU (concurrent streams, other threads) race and must be serialised by
 * the caller.  Allocates nothing: no cudaMalloc, cudaFree or allocating
 * library routine.  The status word of a bounded wait that gave up is not
 * observable through this entry point. */
SWA_API swa_status_t swa_backward_noalloc(const swa_params_t *p, const void *q, const void *k, const void *v,
                                          const void *dy, const void *out, const float *softmax_max,
                                          const float *softmax_sum, const uint8_t *drop_mask, void *dq, void *dk,
                                          void *dv, swa_stream_t stream);

/* Forward + backward of one problem whose tensors live in HOST memory (an
 * addition of this library; the pages' operators take device tensors).  The
 * heads are split into `chunks` equal groups; the first group is split into
 * halves, its first half again, and so on while 2^l * chunks divides N and
 * N_kv (at most three levels), and the last group the same way mirrored, so
 * that less is copied before the first computation and after the last.  Each
 * group is copied to its own compact device tensors inside `device_buffer`,
 * computed (swa_forward, then swa_backward) and copied back, and the copies
 * of the next and the previous group run on internal streams while a group
 * computes.  A group's forward starts once its q, k and v are in, and its
 * out and statistics go back while its backward runs.  Consecutive groups
 * compute on two further internal streams in turn, so one group's kernels
 * may start while the previous group's last CTAs still run; each of those
 * has its own device -> host stream.  The five internal streams and their
 * events are created by the first call in a CUDA context and kept until the
 * process exits; calls in one context share them (their enqueueing is
 * serialised by a lock, and their GPU work runs one call after the other).
 * Heads are independent, so the results equal those of one swa_forward +
 * swa_backward on device copies of the same tensors, bit for bit.
 *   q, k, v, dy   host, p->dtype, shapes and layout as for swa_forward /
 *                 swa_backward; page-locked memory lets the copies overlap
 *   out, softmax_max, softmax_sum, dq, dk, dv
 *                 host, written when `stream` completes
 *   chunks        >= 1, dividing N and N_kv.  Dropout needs dropout_gen = 1
 *                 and chunks = 1: there is no drop_mask argument, and the
 *                 generated keep bits are indexed by the whole problem's heads
 *   device_buffer device, >= swa_step_host_buffer_size bytes, 256-byte aligned
 * All work is enqueued behind the work already on `stream`, and `stream`
 * completes only once every result is in host memory.  Errors: those of
 * swa_forward / swa_backward, SWA_ERR_PARAM_INVALID (chunks), and
 * SWA_ERR_CUDA.  On an error part of the work may already be enqueued;
 * `stream` then still completes only after every copy enqueued by the call
 * has run, so the host buffers may be released once it has. */
SWA_API swa_status_t swa_step_host_buffer_size(const swa_params_t *p, int chunks, size_t *bytes);
SWA_API swa_status_t swa_step_host(const swa_params_t *p, int chunks, const void *q, const void *k,
                                   const void *v, const void *dy, void *out, float *softmax_max,
                                   float *softmax_sum, void *dq, void *dk, void *dv, void *device_buffer,
                                   size_t device_bytes, swa_stream_t stream);
/* swa_workspace_status over every chunk's forward and backward workspace
 * inside a swa_step_host device_buffer. */
SWA_API swa_status_t swa_step_host_status(const swa_params_t *p, int chunks, const void *device_buffer,
                                          swa_stream_t stream);

/* Write the keep mask that p->dropout_seed / p->dropout_offset stand for
 * (see "Dropout" above) in the drop_mask layout: ceil(bits / 8) bytes, bits =
 * sum over sequences of N * Sq_b * Skv_b.  mask is device memory of
 * mask_bytes bytes; bytes past the last element are zero.  It lets a caller
 * keep or inspect the mask a seed-driven call used; the pages' low-level
 * backward takes it as drop_mask.  Errors: the size query's,
 * SWA_ERR_PARAM_NULLPTR, SWA_ERR_WORKSPACE (mask_bytes too small),
 * SWA_ERR_CUDA. */
SWA_API swa_status_t swa_dropout_mask(const swa_params_t *p, uint8_t *mask, size_t mask_bytes,
                                      swa_stream_t stream);

/* Wait for `stream`, then report whether any kernel of the last call that
 * used `workspace` gave up a bounded wait: SWA_OK or SWA_ERR_TIMEOUT
 * (SWA_ERR_CUDA if the stream itself failed).  In the bounds-checked build
 * (compiled with SWA_CHECKS = 1; its kernels test every global load and
 * store against the extent of its tensor and skip it when outside) a
 * skipped access reports SWA_ERR_BOUNDS. */
SWA_API swa_status_t swa_workspace_status(const void *workspace, swa_stream_t stream);

/* Measurement support.  `events` is NULL (stop recording) or an array of
 * eight cudaEvent_t handles owned by the caller: {forward start, forward
 * stop, dK/dV start, dK/dV stop, dQ start, dQ stop, preprocess start,
 * preprocess stop}.  Later calls on this thread record each pair on their
 * stream immediately around the corresponding kernel launch (swa_forward's
 * forward kernel; swa_backward's key-major dK/dV kernel, query-major dQ
 * kernel and D / lse2 preprocess).  No other effect. */
SWA_API void swa_set_timing_events(void *const *events);

/* Test and inspection support (additions of this library; the pages have no
 * counterpart).
 *
 * swa_debug_schedule: the work items that the band / varlen tile scheduler
 * hands to the kernels of one pass, computed on the host by the same code
 * the kernels run (no GPU needed).  The window is the BAND inequality of the
 * FlashAttentionVarLenScore doc (preTokens / nextTokens as the left and right
 * edges): a 128-row query tile touches one run of 128-row key tiles and a
 * key tile one run of query tiles; tiles outside the runs are skipped.
 *   pass 0   query-major dQ pass (and the forward one CTA per query tile):
 *            one item per query tile of each (batch, query head); partners
 *            are key tiles
 *   pass 1   key-major dK / dV pass: one item per key tile of each (batch,
 *            key/value head); partners are query tiles, walked for every
 *            query head of the group
 *   pass 2   the forward one CTA per pair of query tiles (D <= 64, when the
 *            pairs fill every SM): one item per pair p (query tiles 2p and
 *            2p + 1) of each (batch, query head); partners are the key tiles
 *            from the first start to the last end of the two tiles' runs
 *   items    host, 6 int32 per item in launch order: launch index, batch,
 *            head, tile, first partner tile, partner tile count; at most
 *            `capacity` items are written (items may be NULL to count)
 *   count    host, receives the number of items
 * Errors: the size query's, SWA_ERR_PARAM_NULLPTR (count), and
 * SWA_ERR_PARAM_INVALID (pass).
 *
 * swa_debug_stall: while `kernels` is non-zero, every later call makes the
 * compute warps of the selected kernels (bit 0 forward, bit 1 key-major
 * dK / dV, bit 2 query-major dQ) first wait on a barrier that nothing
 * completes.  That wait gives up after its 2 s limit like any other, the
 * kernel drains its copies and tensor-core work in flight, frees its tensor
 * memory and returns, and swa_workspace_status then reports
 * SWA_ERR_TIMEOUT: it exercises the bounded-wait failure path without a
 * fault.  The outputs of such a call are undefined.  Process-wide; 0 turns
 * it off.
 *
 * swa_debug_forward_pairs: how later forward calls with D <= 64 pick their
 * kernel.  0 (the default): one CTA per pair of query tiles when the pairs
 * fill every SM at least once, else one CTA per query tile; 1: always pairs;
 * 2: never.  Both kernels compute the same results; the switch lets tests
 * reach each on small problems.  Process-wide.
 *
 * swa_debug_extent_slack: every later call takes `elems` (>= 0; negative
 * values count as 0) off each tensor extent that the bounds-checked build
 * (libswa_checked.so, see swa_workspace_status) tests the kernels' global
 * loads and stores against, so that accesses at the end of q / out / dQ,
 * k / dK / dV, the statistics and a stored keep mask count as outside their
 * tensor: they are skipped and the call's status word reports
 * SWA_ERR_BOUNDS.  It exercises that path with accesses that are all in
 * range.  The release build has no such checks and ignores it; the
 * outputs of a call it affects are undefined.  Process-wide; 0 turns it off. */
SWA_API swa_status_t swa_debug_schedule(const swa_params_t *p, int32_t pass, int32_t *items, int64_t capacity,
                                        int64_t *count);
SWA_API void swa_debug_stall(int32_t kernels);
SWA_API void swa_debug_forward_pairs(int32_t mode);
SWA_API void swa_debug_extent_slack(int64_t elems);

/* Text describing the last non-OK status returned on this thread. */
SWA_API const char *swa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SWA_H */
