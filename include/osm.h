/*
 * osm.h — C ABI of libosm: exact softmax attention by the online-softmax
 * recurrence, for one NVIDIA GB300 GPU (sm_103a).
 *
 * The operations follow three web pages on one subject:
 *   [P1] "Online Softmax: How FlashAttention Skips the N×N Matrix" (dev.to)
 *   [P2] "Online softmax" (guide.dupenodi.dev)
 *   [P3] "Online softmax" (zerotofrontier.app, chapter 12.2)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is DEVICE memory owned by the caller.  The library
 *    never allocates, frees or synchronises; it only launches kernels.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Outputs are ready when the stream reaches that point.
 *  - Tensors are dense and contiguous, row-major, innermost dimension last.
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns OSM_ERR_INVALID_VALUE (or OSM_ERR_UNSUPPORTED for a valid
 *    but unimplemented case) and launches nothing.  Sequence lengths (Nq, Nk)
 *    above 2^30 are unsupported.  A failed launch returns
 *    OSM_ERR_CUDA.  No call aborts the process or throws.
 *  - Scores are s = scale * (q . k).  Log-sum-exp outputs are natural-log
 *    values of the scaled scores.  Kernels work in base 2 internally (log2(e)
 *    is folded into the scale once) and convert back ([P3] "Precision").
 *  - A query row with no visible key (a fully masked row) gets output 0 and
 *    log-sum-exp -inf ([P3] "Precision": such a row ends with l = 0 and is
 *    handled explicitly; its summary is the merge identity (-inf, 0, 0)).
 *  - Device-side waits are bounded.  If one runs out, the kernel records an
 *    error word, drains its own copies and returns; osm_device_status()
 *    reports it.  Outputs of that launch are then undefined.
 */
#ifndef OSM_H_
#define OSM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *osm_stream_t; /* same type as cudaStream_t */

typedef enum {
  OSM_OK = 0,
  OSM_ERR_INVALID_VALUE = 1, /* null pointer, bad size, misalignment, small workspace */
  OSM_ERR_UNSUPPORTED = 2,   /* valid request this build does not implement (e.g. d) */
  OSM_ERR_CUDA = 3,          /* a CUDA launch or runtime call failed */
  OSM_ERR_TIMEOUT = 4,       /* a bounded device-side wait ran out (osm_device_status) */
  OSM_ERR_CONFLICT = 5,      /* two forward launches in flight shared a work-item
                                counter (osm_device_status; see osm_attn_fwd) */
  OSM_ERR_INDEX = 6          /* a build with OSM_CHECKED found a global index out of
                                range and skipped the access (osm_device_status) */
} osm_status;

typedef enum { OSM_F32 = 0, OSM_BF16 = 1 } osm_dtype;

/*
 * osm_softmax_rows — softmax of every row of an fp32 matrix.
 *
 * Defines: y[r, i] = exp(x[r, i] - m_r) / l_r with m_r the row maximum and
 * l_r = sum_i exp(x[r, i] - m_r)  ([P3] "Three passes, and why that is a
 * problem").  Computed with the online normaliser ([P3] "The recurrence, and
 * a proof that it is right"): per-thread (m, l) summaries merged exactly
 * ([P3] "Merging partial results"), then one scaling pass.  Each element is
 * read from HBM once and written once.
 *
 *   x     [rows, cols] fp32, device, read only.
 *   y     [rows, cols] fp32, device; may equal x (in place); must not
 *         otherwise overlap x.
 *   rows, cols >= 0 (rows * cols == 0 is a no-op returning OSM_OK).
 * Entries must be finite or -inf.  An all -inf row gives zeros.
 * Fast path: x, y 16-byte aligned, cols % 4 == 0, cols <= 131072; any other
 * shape runs a generic two-pass kernel (x read twice, y written once).  On
 * the fast path the thread blocks of a row exchange their summaries through
 * distributed shared memory under a bounded wait; one that runs out records
 * a site (top byte 0x03) that osm_device_status reports as OSM_ERR_TIMEOUT.
 */
osm_status osm_softmax_rows(const float *x, float *y, int64_t rows, int64_t cols,
                            osm_stream_t stream);

/*
 * osm_softmax_topk — the k largest entries of every row of an fp32 matrix and
 * their softmax probabilities, fused: the row comes from HBM once.
 *
 * Defines ([P3] the `softmax_topk` exercise after "Precision, and what can
 * still go wrong", Milakov & Gimelshein's fused softmax + top-k): for row r,
 * idx[r, 0..k-1] are the columns of the k largest x[r, :], in the order
 * larger value first, equal values by smaller column (a total order, so the
 * result is unique), and prob[r, t] = exp(x[r, idx[r, t]] - m_r) / l_r with
 * the row's (m_r, l_r) as in osm_softmax_rows.  A thread-block cluster takes
 * a row: a first sweep over each block's slice forms the online normaliser
 * (m, l) and a threshold that at least k entries reach; a second sweep (the
 * slice is still in L2) keeps, per warp, a running sorted list of the best
 * (value, column) pairs above that threshold.  Normalisers and lists merge
 * exactly in any grouping ([P3] "Merging partial results"), warp by warp,
 * then across the cluster.
 *
 *   x     [rows, cols] fp32, device, read only; entries finite or -inf.
 *   idx   [rows, k] int32 (written);  prob [rows, k] fp32 (written).
 *   rows >= 0 (0 is a no-op), 1 <= k <= cols; k <= 32 (larger k returns
 *   OSM_ERR_UNSUPPORTED: a warp's list holds 32 pairs, one per lane); cols <= 2^31 - 1;
 *   rows <= 2^28.
 * An all -inf row gives idx = 0..k-1 and prob = 0.  x, idx, prob 4-byte
 * aligned; 16-byte aligned x with cols % 4 == 0 takes the vector-load path.
 */
osm_status osm_softmax_topk(const float *x, int64_t rows, int64_t cols, int k, int32_t *idx,
                            float *prob, osm_stream_t stream);

/*
 * osm_attn_fwd — exact softmax attention forward, BF16 in, FP32 state.
 *
 * Defines: for every (b, h) and query row i,
 *   s_ij = scale * (q_i . k_j),  masked to -inf where j >= key_len[b] or
 *          (causal and j > i + (Nk - Nq))   (causal is bottom-right aligned),
 *   o_i = softmax(s_i) V,   lse_i = log sum_j exp(s_ij).
 * Computed tile by tile ([P3] "Blocks, the bridge to FlashAttention"): 128
 * query rows against streamed 128-key tiles, a running reference m, running
 * sum l and unnormalised output O~ in FP32, rescaled by 2^(m_old - m_new)
 * when the reference moves, masks applied inside the tile loop ([P2] "Walking
 * through it"), one division at the end, lse = m + log l ([P3] "From weights
 * to outputs").  The reference need not be the running maximum ([P3]
 * "Precision, and what can still go wrong": any bound will do); the kernel
 * moves it only when a term would exceed 2^16 or all terms so far underflow.
 * No score matrix is written to memory.
 * Work is handed to the thread blocks through a library-owned counter that
 * the call resets on `stream` (two 4-byte fills, then the kernel): count 0
 * and the launch's own tag.  Calls on different streams may overlap as long
 * as fewer than 1024 direct calls (and, separately, 1024 captured-graph
 * launches) are in flight at once.  If more are, a launch whose counter was
 * reset by a later one finds a foreign tag when it next draws work, stops
 * drawing and records OSM_ERR_CONFLICT for osm_device_status: its outputs are
 * then wrong (and so may the later launch's be), but not silently.  A launch
 * captured into a CUDA graph keeps its counter and tag for every replay, so
 * two instantiations of one captured forward (or two replays of one graph on
 * different streams) must not run at the same time: they share a counter
 * without the tag telling them apart.
 *
 *   q     [B, H, Nq, d] bf16;  k, v [B, H, Nk, d] bf16 (read only).
 *   o     [B, H, Nq, d] bf16 (written);  lse [B, H, Nq] fp32 (written).
 *   d     64 or 128 (other values return OSM_ERR_UNSUPPORTED).
 *   scale finite and > 0 (e.g. 1/sqrt(d)).
 *   causal 0 or 1.
 *   key_len device int32[B] (valid keys per batch entry, clamped to [0, Nk]
 *         on the device) or NULL for "all Nk keys valid".
 *   B, H, Nq >= 0 (a zero makes the call a no-op), Nk >= 0.
 *   q, k, v, o must be 16-byte aligned; lse 4-byte aligned.
 * Keys past key_len are never allowed into the running sums; their K/V
 * contents must be finite (a NaN/Inf there would poison the tensor-core dot
 * products of the same tile) but otherwise do not affect the result.
 */
osm_status osm_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                        int B, int H, int Nq, int Nk, int d, float scale, int causal,
                        const int32_t *key_len, osm_stream_t stream);

/*
 * osm_attn_fwd_bounded — osm_attn_fwd for scores with a known upper bound.
 *
 * [P3] "Precision, and what can still go wrong": any number at least as large
 * as every score prevents overflow, so with a bound known in advance (for
 * example queries and keys normalised by QK-norm, so |s| <= scale |q| |k|) it
 * can be subtracted once and the running maximum is never needed.  Every row
 * starts from `score_bound` (scaled-score units, natural log) instead of 0.
 * With a valid bound the reference moves only in three cases: when every
 * term so far would underflow (the bound lies more than about 87, 2^126 in
 * weight, above a row's scores: the pages' warning that a loose bound risks
 * underflowing every term), the kernel lowers it; a score above the bound by
 * more than 16 binades' worth raises it; and a chunk of keys after the first
 * tile that outweighs everything before it in the row moves it to that
 * chunk's maximum (lowering it by at most 120 binades), so that a dominant
 * term has weight exactly 1.  The first tile's terms, taken against the bound,
 * enter the divisor as rounded to bf16.  Either way the result is exact to
 * rounding; the bound only decides how often a chunk is redone.
 *
 * Arguments as osm_attn_fwd, plus:
 *   score_bound  finite, |score_bound| <= 1e30 (else OSM_ERR_INVALID_VALUE).
 */
osm_status osm_attn_fwd_bounded(const void *q, const void *k, const void *v, void *o,
                                float *lse, int B, int H, int Nq, int Nk, int d, float scale,
                                int causal, const int32_t *key_len, float score_bound,
                                osm_stream_t stream);

/*
 * osm_attn_fwd_normalised — osm_attn_fwd computed in the normalised form.
 *
 * [P3] "From weights to outputs" writes the same recurrence a second way, the
 * form of the original FlashAttention: keep the output normalised after every
 * key block, o_new = (l_old e^{m_old - m_new} o + sum_j e^{s_j - m_new} v_j)
 * / l_new, one division per block instead of one at the end, and calls the
 * per-block division wasted work.  This entry point computes that form (the
 * tile's weights are divided by the new l before the P V product and the
 * accumulator is scaled by l_old / l_new) so that its cost can be measured
 * against osm_attn_fwd.  Results agree with osm_attn_fwd to rounding; the
 * weights are rounded to bf16 twice (as e^{s - m}, then divided by l), so a
 * row concentrated on a few keys is off by up to twice the bf16 unit
 * roundoff of its weights.
 *
 * Arguments, layouts and errors as osm_attn_fwd.
 */
osm_status osm_attn_fwd_normalised(const void *q, const void *k, const void *v, void *o,
                                   float *lse, int B, int H, int Nq, int Nk, int d, float scale,
                                   int causal, const int32_t *key_len, osm_stream_t stream);

/*
 * osm_attn_bwd — gradients of exact softmax attention, BF16 in and out.
 *
 * Defines ([P3] "From weights to outputs": the log-sum-exp is all the
 * backward pass needs to rebuild the weights, y_j = exp(s_j - lse)): with s,
 * the masks and lse as in osm_attn_fwd, P = exp(s - lse) (0 where masked),
 * and dO the gradient of O,
 *   dV = P^T dO,   dP = dO V^T,   D_i = sum_c dO_ic O_ic,
 *   dS = P * (dP - D_i),   dQ = scale dS K,   dK = scale dS^T Q.
 * The weights are rebuilt tile by tile from q, k and lse; no score matrix is
 * stored.  Three launches on `stream`: D (into the workspace), dK and dV (one
 * CTA per 128-key tile), dQ (one CTA per 128-query tile).
 *
 *   q [B, H, Nq, d], k, v [B, H, Nk, d], o and dout [B, H, Nq, d]: bf16, read only
 *         (o and lse as written by osm_attn_fwd for the same inputs).
 *   lse   [B, H, Nq] fp32, natural log (-inf for a row with no visible key).
 *   dq [B, H, Nq, d], dk, dv [B, H, Nk, d]: bf16, written.
 *   d, scale, causal, key_len: as osm_attn_fwd.  Keys past key_len get
 *         dK = dV = 0.
 *   workspace >= osm_attn_bwd_workspace_bytes(B, H, Nq) bytes of device
 *         memory, 256-byte aligned (holds D, fp32 [B, H, Nq]).
 *   q, k, v, o, dout, dq, dk, dv 16-byte aligned.
 */
size_t osm_attn_bwd_workspace_bytes(int B, int H, int Nq);
osm_status osm_attn_bwd(const void *q, const void *k, const void *v, const void *o,
                        const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                        int H, int Nq, int Nk, int d, float scale, int causal,
                        const int32_t *key_len, void *workspace, size_t workspace_bytes,
                        osm_stream_t stream);

/*
 * osm_attn_decode_splitkv_workspace_bytes — bytes of device workspace that
 * osm_attn_decode_splitkv needs for these sizes (0 if a size is invalid).
 *
 * Workspace layout (fp32, R = B*H rows, S = num_splits), each section starting
 * on a 256-byte boundary:
 *   m  [S][R]      running max of split s for row r (natural-log units)
 *   l  [S][R]      sum over the split of exp(s_j - m)
 *   o~ [S][R][d]   sum over the split of exp(s_j - m) v_j
 * Section offsets: m at 0, l at A, o~ at 2A with A = round_up(4*S*R, 256).
 * An empty split holds the merge identity (-inf, 0, 0).
 */
size_t osm_attn_decode_splitkv_workspace_bytes(int B, int H, int d, int num_splits);

/*
 * osm_attn_decode_splitkv — one query per (b, h) against a long KV cache,
 * with the keys split into num_splits pieces processed by separate thread
 * blocks, each piece summarised as (m, l, o~), then merged exactly
 * ([P3] "Merging partial results" and "The same merge, in log-sum-exp form":
 * Flash-Decoding splits one query's keys across thread blocks and merges).
 *
 *   dt    OSM_BF16 (q, k, v, o in bf16) or OSM_F32 (all fp32).
 *   q     [B, H, 1, d];  k, v [B, H, Nk, d];  o [B, H, 1, d] in dt.
 *   lse   [B, H] fp32.
 *   d     64 or 128.
 *   key_len device int32[B] (clamped to [0, Nk]) or NULL (= Nk).
 *   num_splits 1..256.  Split s of batch entry b covers keys
 *         [s*c, min((s+1)*c, L_b)) with c = ceil(L_b / num_splits), so the
 *         valid length, not Nk, is divided; keys past L_b are never read.
 *   workspace >= osm_attn_decode_splitkv_workspace_bytes(B, H, d, num_splits)
 *         bytes of device memory, 256-byte aligned, owned by the caller; it
 *         holds the per-split summaries (layout above) after the call.
 *   q, k, v, o 16-byte aligned.
 * Two launches on `stream`: the split kernel, then the merge kernel.
 */
osm_status osm_attn_decode_splitkv(osm_dtype dt, const void *q, const void *k, const void *v,
                                   void *o, float *lse, int B, int H, int Nk, int d,
                                   float scale, const int32_t *key_len, int num_splits,
                                   void *workspace, size_t workspace_bytes,
                                   osm_stream_t stream);

/*
 * osm_lse_merge — merge S normalised partial results per row in
 * log-sum-exp form ([P3] "The same merge, in log-sum-exp form"):
 *   lse = log sum_s exp(lse_s),   o = sum_s exp(lse_s - lse) o_s.
 * A part with lse_s = -inf has weight 0; a row whose parts are all -inf gets
 * o = 0, lse = -inf.  Parts are merged in the fixed order s = 0 .. S-1.
 *
 *   o_parts   [S][rows][d] fp32, 16-byte aligned.
 *   lse_parts [S][rows] fp32.
 *   S 1..1024;  rows >= 0;  d 64 or 128.
 *   out_dt    dtype of o: OSM_F32 or OSM_BF16.
 *   o [rows][d] (out_dt), lse [rows] fp32.
 */
osm_status osm_lse_merge(const float *o_parts, const float *lse_parts, int S, int64_t rows,
                         int d, osm_dtype out_dt, void *o, float *lse, osm_stream_t stream);

/*
 * OSM_NOALLOC_SCRATCH_BYTES — size of the device scratch area that libosm
 * reserves (as a fixed-size device array, on every GPU that loads the library,
 * until the process exits) for osm_attn_decode_splitkv_noalloc.
 */
#define OSM_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * osm_attn_decode_splitkv_noalloc — osm_attn_decode_splitkv for callers that
 * cannot allocate device memory.  The pages have no counterpart; this entry
 * point exists for the caller, not for the method.
 *
 * Some callers cannot call cudaMalloc: a plug-in loaded into a host program
 * that owns every byte of device memory and hands its plug-ins no allocator,
 * or code that runs under a fixed device-memory budget where allocating after
 * start-up is forbidden.  Such a caller cannot provide the split summaries'
 * workspace, so this entry point keeps them in a scratch area inside the
 * library instead (OSM_NOALLOC_SCRATCH_BYTES, reserved when the library's
 * device code is loaded).  It calls no allocator of any kind.
 *
 * Arguments, layouts, results and errors are those of osm_attn_decode_splitkv
 * without `workspace` / `workspace_bytes`.  In addition it returns
 * OSM_ERR_INVALID_VALUE, launching nothing, when the summaries would need more
 * than OSM_NOALLOC_SCRATCH_BYTES, i.e. when
 * osm_attn_decode_splitkv_workspace_bytes(B, H, d, num_splits) is larger.
 *
 * The first call on a device looks up the scratch area's device address
 * (with that device current) and caches it with the id of the device's
 * current context; make that first call before any stream capture begins.
 * A call that finds a different context current (after cudaDeviceReset, or
 * under a context the caller created) looks the address up again, so it too
 * should come before any capture.
 * Every call on a device shares the one scratch area, which keeps the last
 * call's summaries; nothing in it needs to start at zero, because the split
 * kernel writes every summary slot that the merge kernel reads.  Calls whose
 * work overlaps on the GPU (on different streams, or from different threads)
 * race on the scratch area and give undefined results: order them on one
 * stream or synchronise between them.
 */
osm_status osm_attn_decode_splitkv_noalloc(osm_dtype dt, const void *q, const void *k,
                                           const void *v, void *o, float *lse, int B, int H,
                                           int Nk, int d, float scale, const int32_t *key_len,
                                           int num_splits, osm_stream_t stream);

/*
 * osm_attn_decode_append — extend each query's stored running summary by
 * newly appended keys, and return the attention output over every key seen.
 *
 * Defines: for each (b, h) with query q = q[b, h, 0], the caller keeps the
 * summary (m, l, o~) of the keys already seen: m = max s_j, l = sum_j
 * exp(s_j - m), o~ = sum_j exp(s_j - m) v_j over those keys ([P3] "Merging
 * partial results"; the empty set's summary is the identity (-inf, 0, 0)).
 * Appending keys is one more step of the recurrence ([P1] "How does this
 * connect to KV-cache decoding?"): the call forms the summary of the keys
 * [key_start[b], key_end[b]) of k, v and merges it into the stored one
 * ([P3] "Merging partial results", property 3: one step is a merge), so after
 * the call the state is the summary of old keys and new keys together, and
 *   o[b, h] = o~ / l,   lse[b, h] = m + log l   (0 and -inf while l = 0).
 * The result equals attention over the union up to rounding, whatever the
 * number and sizes of the appends.
 *
 * Work: the new keys are split as in osm_attn_decode_splitkv (range
 * [key_start, key_end) divided into num_splits equal chunks); the thread block
 * that finishes a row last (counted with an atomic ticket, no device wait)
 * merges the row's split summaries into the state, in the fixed order
 * state, split 0 .. num_splits - 1.  One memset (the tickets) and one kernel
 * on `stream`.
 *
 *   dt         OSM_BF16 (q, k, v, o bf16) or OSM_F32 (all fp32).
 *   q          [B, H, 1, d];  k, v [B, H, Nk, d] (e.g. a KV cache of capacity Nk).
 *   key_start  device int32[B] or NULL (= 0); key_end device int32[B] or NULL
 *              (= Nk).  key_end is clamped to [0, Nk] and key_start to
 *              [0, key_end]; an empty range leaves the state unchanged.
 *   state_m    [B, H] fp32, natural-log units of the scaled scores (-inf: no key yet).
 *   state_l    [B, H] fp32.   state_o [B, H, d] fp32 (unnormalised).
 *              Read and rewritten in place; start from (-inf, 0, 0).
 *   o          [B, H, 1, d] in dt, or NULL;  lse [B, H] fp32, or NULL.
 *   d 64 or 128;  num_splits 1..256;  q, k, v 16-byte aligned.
 *   workspace  >= osm_attn_decode_append_workspace_bytes(B, H, d, num_splits)
 *              bytes, 256-byte aligned: the split summaries (the layout of
 *              osm_attn_decode_splitkv's workspace) followed by B*H tickets.
 * Launches on one stream must not share a workspace or a state concurrently.
 */
size_t osm_attn_decode_append_workspace_bytes(int B, int H, int d, int num_splits);
osm_status osm_attn_decode_append(osm_dtype dt, const void *q, const void *k, const void *v,
                                  int B, int H, int Nk, int d, float scale,
                                  const int32_t *key_start, const int32_t *key_end,
                                  float *state_m, float *state_l, float *state_o, void *o,
                                  float *lse, int num_splits, void *workspace,
                                  size_t workspace_bytes, osm_stream_t stream);

/* Text for a status code (static storage; never NULL). */
const char *osm_status_string(osm_status status);

/*
 * osm_device_status — synchronise `stream`, then read and clear the current
 * device's error word that bounded waits write.  *word = 0 means no device
 * wait ran out since the last call; otherwise it identifies the site: a
 * word whose top byte is 0x0C is a shared work-item counter (return value
 * OSM_ERR_CONFLICT), 0x0E an index found out of range by a build compiled
 * with OSM_CHECKED (OSM_ERR_INDEX; such a build checks the global indices
 * its kernels compute and skips an access that would leave its tensor), any
 * other a bounded wait that ran out (OSM_ERR_TIMEOUT).
 * Returns OSM_ERR_CUDA if the synchronisation itself fails.  Not a hot-path
 * call.
 */
osm_status osm_device_status(osm_stream_t stream, uint32_t *word);

/*
 * osm_selftest_bounded_wait — exercise the failure path of the kernels'
 * bounded waits: one thread waits on a barrier that nothing completes.  The
 * wait gives up after its limit (about one second), records the site code
 * 0x7f0000a1 in the device error word and the kernel exits normally; the next
 * osm_device_status returns OSM_ERR_TIMEOUT with that word.  The device
 * context stays usable.  Not a hot-path call; for tests of error reporting.
 */
osm_status osm_selftest_bounded_wait(osm_stream_t stream);

/* ABI version of this header (major * 100 + minor). */
int osm_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* OSM_H_ */
