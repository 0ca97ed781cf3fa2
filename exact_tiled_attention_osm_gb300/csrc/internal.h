// internal.h — launchers shared between the C-ABI front end (api.cu) and the
// kernel translation units.  Arguments are already validated by the caller.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "osm.h"

namespace osm {

int sm_count_current_device();

// softmax_rows.cu
cudaError_t launch_softmax_rows(const float* x, float* y, int64_t rows, int64_t cols,
                                cudaStream_t s);

// softmax_topk.cu
cudaError_t launch_softmax_topk(const float* x, int64_t rows, int64_t cols, int k, int32_t* idx,
                                float* prob, cudaStream_t s);

// attn_fwd.cu
cudaError_t launch_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int H, int Nq, int Nk, int d, float scale, int causal,
                            const int32_t* key_len, float score_bound, bool normalised,
                            cudaStream_t s, bool* tmap_ok);
cudaError_t read_and_clear_device_error(cudaStream_t s, uint32_t* word);
// decode.cu: the index-check word of a build compiled with OSM_CHECKED
cudaError_t read_and_clear_decode_check(uint32_t* word);
// softmax_rows.cu: the row-softmax kernels' error word (a summary wait that ran out)
cudaError_t read_and_clear_softmax_error(uint32_t* word);
cudaError_t launch_bounded_wait_selftest(cudaStream_t s);

// attn_bwd.cu
size_t attn_bwd_workspace_bytes(int B, int H, int Nq);
cudaError_t launch_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dout, void* dq, void* dk, void* dv,
                            int B, int H, int Nq, int Nk, int d, float scale, int causal,
                            const int32_t* key_len, void* workspace, cudaStream_t s,
                            bool* tmap_ok);
cudaError_t read_and_clear_bwd_error(uint32_t* word);

// decode.cu
size_t decode_workspace_bytes(int B, int H, int d, int S);
cudaError_t launch_decode_splitkv(osm_dtype dt, const void* q, const void* k, const void* v,
                                  void* o, float* lse, int B, int H, int Nk, int d, float scale,
                                  const int32_t* key_len, int S, void* ws, cudaStream_t s);
// the same decode, with the summaries in the library's own scratch area
cudaError_t launch_decode_splitkv_noalloc(osm_dtype dt, const void* q, const void* k,
                                          const void* v, void* o, float* lse, int B, int H,
                                          int Nk, int d, float scale, const int32_t* key_len,
                                          int S, cudaStream_t s);
// extend stored running summaries by the keys [key_start[b], key_end[b])
size_t decode_append_workspace_bytes(int B, int H, int d, int S);
cudaError_t launch_decode_append(osm_dtype dt, const void* q, const void* k, const void* v,
                                 int B, int H, int Nk, int d, float scale,
                                 const int32_t* key_start, const int32_t* key_end, float* state_m,
                                 float* state_l, float* state_o, void* o, float* lse, int S,
                                 void* ws, cudaStream_t s);
cudaError_t launch_lse_merge(const float* o_parts, const float* lse_parts, int S, int64_t rows,
                             int d, osm_dtype out_dt, void* o, float* lse, cudaStream_t s);

}  // namespace osm
