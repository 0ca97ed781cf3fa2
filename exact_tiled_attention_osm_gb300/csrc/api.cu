// api.cu — the extern "C" entry points declared in include/osm.h: argument
// validation on the host (nothing is launched for a bad request), then the
// launch on the caller's stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <limits>
#include <cstdint>

#include "internal.h"
#include "osm.h"

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline osm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? OSM_OK : OSM_ERR_CUDA; }

}  // namespace

extern "C" {

int osm_abi_version(void) { return 103; }

const char* osm_status_string(osm_status st) {
  switch (st) {
    case OSM_OK: return "OSM_OK: success";
    case OSM_ERR_INVALID_VALUE: return "OSM_ERR_INVALID_VALUE: invalid argument";
    case OSM_ERR_UNSUPPORTED: return "OSM_ERR_UNSUPPORTED: case not implemented by this build";
    case OSM_ERR_CUDA: return "OSM_ERR_CUDA: CUDA launch or runtime error";
    case OSM_ERR_TIMEOUT: return "OSM_ERR_TIMEOUT: a bounded device-side wait ran out";
    case OSM_ERR_CONFLICT:
      return "OSM_ERR_CONFLICT: two forward launches in flight shared a work-item counter";
    case OSM_ERR_INDEX:
      return "OSM_ERR_INDEX: a checked build found a global index out of range";
  }
  return "unknown osm_status";
}

osm_status osm_softmax_rows(const float* x, float* y, int64_t rows, int64_t cols,
                            osm_stream_t stream) {
  if (rows < 0 || cols < 0) return OSM_ERR_INVALID_VALUE;
  if (rows == 0 || cols == 0) return OSM_OK;
  if (!x || !y || !aligned4(x) || !aligned4(y)) return OSM_ERR_INVALID_VALUE;
  if (rows > 0x7fffffffLL || cols > (int64_t{1} << 40)) return OSM_ERR_UNSUPPORTED;
  // y may be x itself; any other overlap is refused
  const uintptr_t xb = reinterpret_cast<uintptr_t>(x), yb = reinterpret_cast<uintptr_t>(y);
  const uintptr_t bytes = static_cast<uintptr_t>(rows) * static_cast<uintptr_t>(cols) * 4u;
  if (xb != yb && xb < yb + bytes && yb < xb + bytes) return OSM_ERR_INVALID_VALUE;
  return from_cuda(osm::launch_softmax_rows(x, y, rows, cols, reinterpret_cast<cudaStream_t>(stream)));
}

osm_status osm_softmax_topk(const float* x, int64_t rows, int64_t cols, int k, int32_t* idx,
                            float* prob, osm_stream_t stream) {
  if (rows < 0 || cols < 0) return OSM_ERR_INVALID_VALUE;
  if (rows == 0) return OSM_OK;
  if (k < 1 || k > cols) return OSM_ERR_INVALID_VALUE;
  if (k > 32) return OSM_ERR_UNSUPPORTED;
  if (cols > 0x7fffffffLL || rows > (int64_t{1} << 28)) return OSM_ERR_UNSUPPORTED;
  if (!x || !idx || !prob || !aligned4(x) || !aligned4(idx) || !aligned4(prob))
    return OSM_ERR_INVALID_VALUE;
  return from_cuda(osm::launch_softmax_topk(x, rows, cols, k, idx, prob,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
// longest sequence (Nq, Nk) accepted: keeps every tile and split count, and
// every length rounded up to a tile, inside int arithmetic
constexpr int kMaxSeq = 1 << 30;

osm_status attn_fwd_checked(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int H, int Nq, int Nk, int d, float scale, int causal,
                            const int32_t* key_len, float score_bound, bool normalised,
                            osm_stream_t stream) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return OSM_ERR_INVALID_VALUE;
  if (causal != 0 && causal != 1) return OSM_ERR_INVALID_VALUE;
  if (!(scale > 0.f) || !std::isfinite(scale)) return OSM_ERR_INVALID_VALUE;
  if (d != 64 && d != 128) return (d > 0) ? OSM_ERR_UNSUPPORTED : OSM_ERR_INVALID_VALUE;
  if (Nq > kMaxSeq || Nk > kMaxSeq) return OSM_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * H * Nq == 0) return OSM_OK;
  if (!q || !o || !lse || (Nk > 0 && (!k || !v))) return OSM_ERR_INVALID_VALUE;
  if (!aligned16(q) || !aligned16(o) || !aligned4(lse)) return OSM_ERR_INVALID_VALUE;
  if (Nk > 0 && (!aligned16(k) || !aligned16(v))) return OSM_ERR_INVALID_VALUE;
  if (key_len && !aligned4(key_len)) return OSM_ERR_INVALID_VALUE;
  if (static_cast<int64_t>(B) * H > 0x7fffffffLL) return OSM_ERR_UNSUPPORTED;
  bool tmap_ok = true;
  cudaError_t e = osm::launch_attn_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, key_len,
                                       score_bound, normalised,
                                       reinterpret_cast<cudaStream_t>(stream), &tmap_ok);
  if (!tmap_ok) return OSM_ERR_UNSUPPORTED;  // shape the TMA descriptor cannot express
  return from_cuda(e);
}
}  // namespace

osm_status osm_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int Nq, int Nk, int d, float scale, int causal,
                        const int32_t* key_len, osm_stream_t stream) {
  return attn_fwd_checked(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, key_len,
                          std::numeric_limits<float>::quiet_NaN(), false, stream);
}

osm_status osm_attn_fwd_normalised(const void* q, const void* k, const void* v, void* o,
                                   float* lse, int B, int H, int Nq, int Nk, int d, float scale,
                                   int causal, const int32_t* key_len, osm_stream_t stream) {
  return attn_fwd_checked(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, key_len,
                          std::numeric_limits<float>::quiet_NaN(), true, stream);
}

osm_status osm_attn_fwd_bounded(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int Nq, int Nk, int d, float scale, int causal,
                                const int32_t* key_len, float score_bound, osm_stream_t stream) {
  if (!std::isfinite(score_bound) || std::fabs(score_bound) > 1e30f) return OSM_ERR_INVALID_VALUE;
  return attn_fwd_checked(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, key_len, score_bound,
                          false, stream);
}

size_t osm_attn_bwd_workspace_bytes(int B, int H, int Nq) {
  if (B < 0 || H < 0 || Nq < 0) return 0;
  return osm::attn_bwd_workspace_bytes(B, H, Nq);
}

osm_status osm_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                        int H, int Nq, int Nk, int d, float scale, int causal,
                        const int32_t* key_len, void* workspace, size_t workspace_bytes,
                        osm_stream_t stream) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return OSM_ERR_INVALID_VALUE;
  if (causal != 0 && causal != 1) return OSM_ERR_INVALID_VALUE;
  if (!(scale > 0.f) || !std::isfinite(scale)) return OSM_ERR_INVALID_VALUE;
  if (d != 64 && d != 128) return (d > 0) ? OSM_ERR_UNSUPPORTED : OSM_ERR_INVALID_VALUE;
  if (Nq > kMaxSeq || Nk > kMaxSeq) return OSM_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * H == 0 || (Nq == 0 && Nk == 0)) return OSM_OK;
  if (Nq > 0 && (!q || !o || !lse || !dout || !dq)) return OSM_ERR_INVALID_VALUE;
  if (Nk > 0 && (!k || !v || !dk || !dv)) return OSM_ERR_INVALID_VALUE;
  if ((q && !aligned16(q)) || (k && !aligned16(k)) || (v && !aligned16(v)) ||
      (o && !aligned16(o)) || (dout && !aligned16(dout)) || (dq && !aligned16(dq)) ||
      (dk && !aligned16(dk)) || (dv && !aligned16(dv)) || (lse && !aligned4(lse)))
    return OSM_ERR_INVALID_VALUE;
  if (key_len && !aligned4(key_len)) return OSM_ERR_INVALID_VALUE;
  if (Nq > 0) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return OSM_ERR_INVALID_VALUE;
    if (workspace_bytes < osm::attn_bwd_workspace_bytes(B, H, Nq)) return OSM_ERR_INVALID_VALUE;
  }
  const int64_t tiles = static_cast<int64_t>(B) * H * ((std::max(Nq, Nk) + 127) / 128);
  if (tiles > 0x7fffffffLL) return OSM_ERR_UNSUPPORTED;
  bool tmap_ok = true;
  cudaError_t e = osm::launch_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, scale,
                                       causal, key_len, workspace,
                                       reinterpret_cast<cudaStream_t>(stream), &tmap_ok);
  if (!tmap_ok) return OSM_ERR_UNSUPPORTED;
  return from_cuda(e);
}

size_t osm_attn_decode_splitkv_workspace_bytes(int B, int H, int d, int num_splits) {
  if (B < 0 || H < 0 || (d != 64 && d != 128) || num_splits < 1 || num_splits > 256) return 0;
  return osm::decode_workspace_bytes(B, H, d, num_splits);
}

osm_status osm_attn_decode_splitkv(osm_dtype dt, const void* q, const void* k, const void* v,
                                   void* o, float* lse, int B, int H, int Nk, int d, float scale,
                                   const int32_t* key_len, int num_splits, void* workspace,
                                   size_t workspace_bytes, osm_stream_t stream) {
  if (dt != OSM_F32 && dt != OSM_BF16) return OSM_ERR_INVALID_VALUE;
  if (B < 0 || H < 0 || Nk < 0) return OSM_ERR_INVALID_VALUE;
  if (d != 64 && d != 128) return (d > 0) ? OSM_ERR_UNSUPPORTED : OSM_ERR_INVALID_VALUE;
  if (num_splits < 1 || num_splits > 256) return OSM_ERR_INVALID_VALUE;
  if (!(scale > 0.f) || !std::isfinite(scale)) return OSM_ERR_INVALID_VALUE;
  if (static_cast<int64_t>(B) * H == 0) return OSM_OK;
  if (B > 65535 || H > 65535 || Nk > kMaxSeq) return OSM_ERR_UNSUPPORTED;
  if (!q || !o || !lse || !workspace || (Nk > 0 && (!k || !v))) return OSM_ERR_INVALID_VALUE;
  if (!aligned16(q) || !aligned16(o) || !aligned4(lse)) return OSM_ERR_INVALID_VALUE;
  if (Nk > 0 && (!aligned16(k) || !aligned16(v))) return OSM_ERR_INVALID_VALUE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return OSM_ERR_INVALID_VALUE;
  if (key_len && !aligned4(key_len)) return OSM_ERR_INVALID_VALUE;
  if (workspace_bytes < osm::decode_workspace_bytes(B, H, d, num_splits))
    return OSM_ERR_INVALID_VALUE;
  return from_cuda(osm::launch_decode_splitkv(dt, q, k, v, o, lse, B, H, Nk, d, scale, key_len,
                                              num_splits, workspace,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

osm_status osm_attn_decode_splitkv_noalloc(osm_dtype dt, const void* q, const void* k,
                                           const void* v, void* o, float* lse, int B, int H,
                                           int Nk, int d, float scale, const int32_t* key_len,
                                           int num_splits, osm_stream_t stream) {
  if (dt != OSM_F32 && dt != OSM_BF16) return OSM_ERR_INVALID_VALUE;
  if (B < 0 || H < 0 || Nk < 0) return OSM_ERR_INVALID_VALUE;
  if (d != 64 && d != 128) return (d > 0) ? OSM_ERR_UNSUPPORTED : OSM_ERR_INVALID_VALUE;
  if (num_splits < 1 || num_splits > 256) return OSM_ERR_INVALID_VALUE;
  if (!(scale > 0.f) || !std::isfinite(scale)) return OSM_ERR_INVALID_VALUE;
  if (static_cast<int64_t>(B) * H == 0) return OSM_OK;
  if (B > 65535 || H > 65535 || Nk > kMaxSeq) return OSM_ERR_UNSUPPORTED;
  // the summaries must fit the library's fixed scratch area
  if (osm::decode_workspace_bytes(B, H, d, num_splits) > OSM_NOALLOC_SCRATCH_BYTES)
    return OSM_ERR_INVALID_VALUE;
  if (!q || !o || !lse || (Nk > 0 && (!k || !v))) return OSM_ERR_INVALID_VALUE;
  if (!aligned16(q) || !aligned16(o) || !aligned4(lse)) return OSM_ERR_INVALID_VALUE;
  if (Nk > 0 && (!aligned16(k) || !aligned16(v))) return OSM_ERR_INVALID_VALUE;
  if (key_len && !aligned4(key_len)) return OSM_ERR_INVALID_VALUE;
  return from_cuda(osm::launch_decode_splitkv_noalloc(dt, q, k, v, o, lse, B, H, Nk, d, scale,
                                                      key_len, num_splits,
                                                      reinterpret_cast<cudaStream_t>(stream)));
}

size_t osm_attn_decode_append_workspace_bytes(int B, int H, int d, int num_splits) {
  if (B < 0 || H < 0 || (d != 64 && d != 128) || num_splits < 1 || num_splits > 256) return 0;
  return osm::decode_append_workspace_bytes(B, H, d, num_splits);
}

osm_status osm_attn_decode_append(osm_dtype dt, const void* q, const void* k, const void* v,
                                  int B, int H, int Nk, int d, float scale,
                                  const int32_t* key_start, const int32_t* key_end,
                                  float* state_m, float* state_l, float* state_o, void* o,
                                  float* lse, int num_splits, void* workspace,
                                  size_t workspace_bytes, osm_stream_t stream) {
  if (dt != OSM_F32 && dt != OSM_BF16) return OSM_ERR_INVALID_VALUE;
  if (B < 0 || H < 0 || Nk < 0) return OSM_ERR_INVALID_VALUE;
  if (d != 64 && d != 128) return (d > 0) ? OSM_ERR_UNSUPPORTED : OSM_ERR_INVALID_VALUE;
  if (num_splits < 1 || num_splits > 256) return OSM_ERR_INVALID_VALUE;
  if (!(scale > 0.f) || !std::isfinite(scale)) return OSM_ERR_INVALID_VALUE;
  if (static_cast<int64_t>(B) * H == 0) return OSM_OK;
  if (B > 65535 || H > 65535 || Nk > kMaxSeq) return OSM_ERR_UNSUPPORTED;
  if (!q || !state_m || !state_l || !state_o || !workspace || (Nk > 0 && (!k || !v)))
    return OSM_ERR_INVALID_VALUE;
  if (!aligned16(q) || !aligned4(state_m) || !aligned4(state_l) || !aligned4(state_o))
    return OSM_ERR_INVALID_VALUE;
  if ((o && !aligned4(o)) || (lse && !aligned4(lse))) return OSM_ERR_INVALID_VALUE;
  if (Nk > 0 && (!aligned16(k) || !aligned16(v))) return OSM_ERR_INVALID_VALUE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return OSM_ERR_INVALID_VALUE;
  if ((key_start && !aligned4(key_start)) || (key_end && !aligned4(key_end)))
    return OSM_ERR_INVALID_VALUE;
  if (workspace_bytes < osm::decode_append_workspace_bytes(B, H, d, num_splits))
    return OSM_ERR_INVALID_VALUE;
  return from_cuda(osm::launch_decode_append(dt, q, k, v, B, H, Nk, d, scale, key_start, key_end,
                                             state_m, state_l, state_o, o, lse, num_splits,
                                             workspace, reinterpret_cast<cudaStream_t>(stream)));
}

osm_status osm_lse_merge(const float* o_parts, const float* lse_parts, int S, int64_t rows, int d,
                         osm_dtype out_dt, void* o, float* lse, osm_stream_t stream) {
  if (out_dt != OSM_F32 && out_dt != OSM_BF16) return OSM_ERR_INVALID_VALUE;
  if (S < 1 || S > 1024 || rows < 0) return OSM_ERR_INVALID_VALUE;
  if (d != 64 && d != 128) return (d > 0) ? OSM_ERR_UNSUPPORTED : OSM_ERR_INVALID_VALUE;
  if (rows == 0) return OSM_OK;
  if (rows * 32 > 0x7fffffffLL * 256LL) return OSM_ERR_UNSUPPORTED;
  if (!o_parts || !lse_parts || !o || !lse) return OSM_ERR_INVALID_VALUE;
  if (!aligned16(o_parts) || !aligned4(lse_parts) || !aligned4(o) || !aligned4(lse))
    return OSM_ERR_INVALID_VALUE;
  return from_cuda(osm::launch_lse_merge(o_parts, lse_parts, S, rows, d, out_dt, o, lse,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

osm_status osm_selftest_bounded_wait(osm_stream_t stream) {
  return from_cuda(osm::launch_bounded_wait_selftest(reinterpret_cast<cudaStream_t>(stream)));
}

osm_status osm_device_status(osm_stream_t stream, uint32_t* word) {
  if (!word) return OSM_ERR_INVALID_VALUE;
  *word = 0;
  cudaError_t e = osm::read_and_clear_device_error(reinterpret_cast<cudaStream_t>(stream), word);
  if (e != cudaSuccess) return OSM_ERR_CUDA;
  uint32_t wb = 0;  // the backward kernels keep their own word
  e = osm::read_and_clear_bwd_error(&wb);
  if (e != cudaSuccess) return OSM_ERR_CUDA;
  if (*word == 0) *word = wb;
  uint32_t wd = 0;  // the decode kernels' index-check word (checked builds)
  e = osm::read_and_clear_decode_check(&wd);
  if (e != cudaSuccess) return OSM_ERR_CUDA;
  if (*word == 0) *word = wd;
  uint32_t ws = 0;  // the row-softmax kernels' word
  e = osm::read_and_clear_softmax_error(&ws);
  if (e != cudaSuccess) return OSM_ERR_CUDA;
  if (*word == 0) *word = ws;
  if (*word == 0) return OSM_OK;
  const uint32_t top = *word >> 24;
  return top == 0x0Cu ? OSM_ERR_CONFLICT : (top == 0x0Eu ? OSM_ERR_INDEX : OSM_ERR_TIMEOUT);
}

}  // extern "C"
