// decode.cu — split-KV decode (one query per (b, h)) and the exact merge of
// partial summaries.
//
// "Online softmax" (zerotofrontier.app): "Merging partial results" defines the
// summary (m, l, o~) of a piece of a row and the merge that combines two
// pieces exactly; "The same merge, in log-sum-exp form" describes
// Flash-Decoding, which splits one query's keys across thread blocks and merges
// the pieces.  "Online Softmax: How FlashAttention Skips the N×N Matrix"
// (dev.to), "How does the online softmax recurrence work?", gives the per-block
// recurrence each warp runs over its keys.
//
// Split kernel: grid (split, h, b), four warps.  Lanes of a warp cover one
// 16-byte slice of a key row each; a warp takes a block of keys per step with
// all its K and V loads in flight at once, forms the scores by a shuffle
// reduction, and updates its running (m, l, o~) with exact rescaling whenever
// the block raises the max.  The four warps' summaries are merged in shared
// memory and the split's summary goes to the workspace.  Keys past the valid
// length are never read.  Merge kernel: one warp per row merges the splits in
// order s = 0 .. S-1.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace osm {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr int kWarps = 4;

__device__ __forceinline__ float rebase2(float m, float mn) {  // base-2 units
  return m == kNegInf ? 0.f : ptx::ex2(m - mn);
}

// element type helpers: unpack one 16-byte slice into EPL floats
template <typename T>
struct Slice;
template <>
struct Slice<__nv_bfloat16> {
  static constexpr int EPL = 8;
  __device__ static __forceinline__ void unpack(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};
template <>
struct Slice<float> {
  static constexpr int EPL = 4;
  __device__ static __forceinline__ void unpack(const uint4& u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
};

template <typename T, int D>
struct Cfg {
  static constexpr int EPL = Slice<T>::EPL;            // elements per lane slice
  static constexpr int LPK = D / EPL;                  // lanes per key row
  static constexpr int KPP = 32 / LPK;                 // keys per warp pass
  static constexpr int R = (KPP >= 4) ? 4 : 8;         // passes per block
  static constexpr int BLOCK = KPP * R;                // keys per warp step
};

struct Workspace {
  float* m;
  float* l;
  float* o;
};

// Index faults found by an OSM_CHECKED build (0x0E02xxxx); read and cleared
// by osm_device_status.
__device__ unsigned int g_chk_word;
constexpr unsigned kChk = 0x0E020000u;
// Running summaries extended in place by the append form of the split kernel.
struct AppendState {
  float* m;               // [rows] natural-log units
  float* l;               // [rows]
  float* o;               // [rows][D] unnormalised
  void* out;              // [rows][D] normalised output (bf16 or fp32), or null
  float* lse;             // [rows], or null
  int out_bf16;
  unsigned int* tickets;  // [rows], zero at launch
};
__host__ __device__ inline size_t ws_section(int64_t n) { return ((n * 4 + 255) / 256) * 256; }

// APPEND: the keys are [key_start[b], key_len[b]) and the CTA that finishes a
// row last (a ticket counter, no waiting) merges the row's split summaries
// into the stored running summary: state <- state (+) split_0 (+) ... (+)
// split_{S-1}, then writes the normalised output.
template <typename T, int D, bool APPEND>
__global__ void __launch_bounds__(kWarps * 32) decode_split_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const int32_t* __restrict__ key_len, int H, int Nk, int S, float scale_log2, Workspace ws,
    const int32_t* __restrict__ key_start, AppendState st) {
  using C = Cfg<T, D>;
  constexpr int EPL = C::EPL, LPK = C::LPK, KPP = C::KPP, R = C::R, BLOCK = C::BLOCK;
  __shared__ float sm_m[kWarps], sm_l[kWarps];
  __shared__ float sm_o[kWarps][D];

  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = lane / LPK;       // which key of a pass this lane works on
  const int sl = lane % LPK;        // which 16-byte slice of the row
  const int64_t row = static_cast<int64_t>(b) * H + h;
  int L = key_len ? key_len[b] : Nk;
  L = L < 0 ? 0 : (L > Nk ? Nk : L);
  int K0 = 0;
  if (APPEND && key_start) K0 = min(max(key_start[b], 0), L);
  const int n = L - K0;
  const int chunk = (n + S - 1) / S;
  const int k_begin = K0 + min(n, s * chunk);
  const int k_end = K0 + min(n, s * chunk + chunk);

  // query slice, pre-multiplied by scale*log2(e) so scores come out in base-2 units
  float qf[EPL];
  {
    const uint4 u = reinterpret_cast<const uint4*>(q + row * D)[sl];
    Slice<T>::unpack(u, qf);
#pragma unroll
    for (int e = 0; e < EPL; ++e) qf[e] *= scale_log2;
  }
  const uint4* kr = reinterpret_cast<const uint4*>(k + row * static_cast<int64_t>(Nk) * D);
  const uint4* vr = reinterpret_cast<const uint4*>(v + row * static_cast<int64_t>(Nk) * D);

  float m = kNegInf, l = 0.f;
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;

  for (int kb = k_begin + warp * BLOCK; kb < k_end; kb += kWarps * BLOCK) {
    uint4 ku[R], vu[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int j = kb + r * KPP + grp;
      if (j < k_end && ptx::checked(j >= 0 && j < Nk, &g_chk_word, kChk | 1)) {
        ku[r] = __ldcs(kr + static_cast<int64_t>(j) * LPK + sl);
        vu[r] = __ldcs(vr + static_cast<int64_t>(j) * LPK + sl);
      } else {
        ku[r] = make_uint4(0, 0, 0, 0);
        vu[r] = make_uint4(0, 0, 0, 0);
      }
    }
    float sc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float kf[EPL];
      Slice<T>::unpack(ku[r], kf);
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) d = fmaf(qf[e], kf[e], d);
#pragma unroll
      for (int off = LPK / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
      sc[r] = (kb + r * KPP + grp < k_end) ? d : kNegInf;
    }
    float mb = sc[0];
#pragma unroll
    for (int r = 1; r < R; ++r) mb = fmaxf(mb, sc[r]);
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
    const float mn = fmaxf(m, mb);  // finite: the block's first key is valid
    const float alpha = rebase2(m, mn);
    float ps = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] *= alpha;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float p = ptx::ex2(sc[r] - mn);
      ps += p;
      float vf[EPL];
      Slice<T>::unpack(vu[r], vf);
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = fmaf(p, vf[e], acc[e]);
    }
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * alpha + ps;
    m = mn;
  }
  // lanes with the same slice but different keys share m: add their outputs
#pragma unroll
  for (int off = LPK; off < 32; off <<= 1) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
  }
  if (lane == 0) {
    sm_m[warp] = m;
    sm_l[warp] = l;
  }
  if (grp == 0) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) sm_o[warp][sl * EPL + e] = acc[e];
  }
  __syncthreads();
  // merge the warps' summaries (fixed order)
  float M = sm_m[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) M = fmaxf(M, sm_m[w]);
  float wgt[kWarps];
  float Lt = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    wgt[w] = rebase2(sm_m[w], M);
    Lt += sm_l[w] * wgt[w];
  }
  const int64_t p = static_cast<int64_t>(s) * gridDim.y * gridDim.z + row;
  if (!ptx::checked(p < static_cast<int64_t>(S) * gridDim.y * gridDim.z, &g_chk_word, kChk | 2)) return;
  for (int c = threadIdx.x; c < D; c += kWarps * 32) {
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) o += sm_o[w][c] * wgt[w];
    ws.o[p * D + c] = o;
  }
  if (threadIdx.x == 0) {
    ws.m[p] = (M == kNegInf) ? kNegInf : M * kLn2;  // natural-log units
    ws.l[p] = Lt;
  }
  if constexpr (APPEND) {
    __shared__ int sm_last;
    __threadfence();  // this split's summary is visible before its ticket is
    __syncthreads();
    if (threadIdx.x == 0) sm_last = atomicAdd(st.tickets + row, 1u) == static_cast<unsigned>(S - 1);
    __syncthreads();
    if (!sm_last) return;
    __threadfence();
    const int64_t R = static_cast<int64_t>(gridDim.y) * gridDim.z;
    // merge in the fixed order: stored summary, then splits 0 .. S-1
    const float m0 = st.m[row];
    float Mg = m0;
    for (int t = 0; t < S; ++t) Mg = fmaxf(Mg, __ldcg(ws.m + t * R + row));
    float lg = 0.f, og = 0.f;
    const int c = threadIdx.x;
    if (Mg != kNegInf) {
      if (m0 != kNegInf) {
        const float w = ptx::ex2((m0 - Mg) * kLog2e);
        lg = st.l[row] * w;
        if (c < D) og = st.o[row * D + c] * w;
      }
      for (int t = 0; t < S; ++t) {
        const float mt = __ldcg(ws.m + t * R + row);
        if (mt == kNegInf) continue;
        const float w = ptx::ex2((mt - Mg) * kLog2e);
        lg = fmaf(__ldcg(ws.l + t * R + row), w, lg);
        if (c < D) og = fmaf(__ldcg(ws.o + (t * R + row) * D + c), w, og);
      }
    }
    if (c < D) {
      st.o[row * D + c] = og;
      if (st.out) {
        const float val = lg > 0.f ? og / lg : 0.f;
        if (st.out_bf16)
          static_cast<__nv_bfloat16*>(st.out)[row * D + c] = __float2bfloat16_rn(val);
        else
          static_cast<float*>(st.out)[row * D + c] = val;
      }
    }
    if (c == 0) {
      st.m[row] = Mg;
      st.l[row] = lg;
      if (st.lse) st.lse[row] = lg > 0.f ? Mg + logf(lg) : kNegInf;
    }
  }
}

template <typename T>
__device__ __forceinline__ void store_out(T* dst, float val);
template <>
__device__ __forceinline__ void store_out<float>(float* dst, float val) {
  *dst = val;
}
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* dst, float val) {
  *dst = __float2bfloat16_rn(val);
}

// One warp per row.  TRIPLE: parts are (m, l, o~) summaries.  Otherwise parts
// are normalised (o_s, lse_s), i.e. the summaries (lse_s, 1, o_s).
template <int D, bool TRIPLE, typename TO>
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ mpart,
                                                    const float* __restrict__ lpart,
                                                    const float* __restrict__ opart, int S,
                                                    int64_t rows, TO* __restrict__ out,
                                                    float* __restrict__ lse) {
  constexpr int PER = D / 32;
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  if (!ptx::checked(S > 0 && lane * PER + PER <= D, &g_chk_word, kChk | 3)) return;
  float M = kNegInf;
  for (int s = 0; s < S; ++s) M = fmaxf(M, mpart[s * rows + row]);
  float l = 0.f, o[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) o[e] = 0.f;
  if (M != kNegInf) {
    for (int s = 0; s < S; ++s) {
      const float ms = mpart[s * rows + row];
      if (ms == kNegInf) continue;
      const float w = ptx::ex2((ms - M) * kLog2e);
      l = fmaf(TRIPLE ? lpart[s * rows + row] : 1.f, w, l);
      const float* src = opart + (s * rows + row) * D + lane * PER;
#pragma unroll
      for (int e = 0; e < PER; ++e) o[e] = fmaf(w, src[e], o[e]);
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int e = 0; e < PER; ++e) store_out<TO>(out + row * D + lane * PER + e, o[e] * inv);
  if (lane == 0) lse[row] = l > 0.f ? M + logf(l) : kNegInf;
}

template <int D, bool TRIPLE>
cudaError_t launch_merge_d(const float* mp, const float* lp, const float* op, int S, int64_t rows,
                           osm_dtype out_dt, void* o, float* lse, cudaStream_t s) {
  const unsigned blocks = static_cast<unsigned>((rows * 32 + 255) / 256);
  if (out_dt == OSM_BF16)
    merge_kernel<D, TRIPLE, __nv_bfloat16>
        <<<blocks, 256, 0, s>>>(mp, lp, op, S, rows, static_cast<__nv_bfloat16*>(o), lse);
  else
    merge_kernel<D, TRIPLE, float>
        <<<blocks, 256, 0, s>>>(mp, lp, op, S, rows, static_cast<float*>(o), lse);
  return cudaGetLastError();
}

template <bool TRIPLE>
cudaError_t launch_merge(const float* mp, const float* lp, const float* op, int S, int64_t rows,
                         int d, osm_dtype out_dt, void* o, float* lse, cudaStream_t s) {
  if (d == 128) return launch_merge_d<128, TRIPLE>(mp, lp, op, S, rows, out_dt, o, lse, s);
  return launch_merge_d<64, TRIPLE>(mp, lp, op, S, rows, out_dt, o, lse, s);
}

Workspace carve(void* ws, int64_t n_parts, int d) {
  char* p = static_cast<char*>(ws);
  const size_t a = ws_section(n_parts);
  return Workspace{reinterpret_cast<float*>(p), reinterpret_cast<float*>(p + a),
                   reinterpret_cast<float*>(p + 2 * a)};
}

}  // namespace

size_t decode_workspace_bytes(int B, int H, int d, int S) {
  const int64_t n = static_cast<int64_t>(B) * H * S;
  return 2 * ws_section(n) + static_cast<size_t>(n) * d * 4;
}

cudaError_t launch_decode_splitkv(osm_dtype dt, const void* q, const void* k, const void* v,
                                  void* o, float* lse, int B, int H, int Nk, int d, float scale,
                                  const int32_t* key_len, int S, void* ws_ptr, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(B) * H;
  Workspace ws = carve(ws_ptr, rows * S, d);
  const float sl2 = scale * kLog2e;
  const dim3 grid(S, H, B), block(kWarps * 32);
  if (dt == OSM_BF16) {
    using T = __nv_bfloat16;
    if (d == 128)
      decode_split_kernel<T, 128, false><<<grid, block, 0, s>>>(
          static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), key_len,
          H, Nk, S, sl2, ws, nullptr, AppendState{});
    else
      decode_split_kernel<T, 64, false><<<grid, block, 0, s>>>(
          static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), key_len,
          H, Nk, S, sl2, ws, nullptr, AppendState{});
  } else {
    using T = float;
    if (d == 128)
      decode_split_kernel<T, 128, false><<<grid, block, 0, s>>>(
          static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), key_len,
          H, Nk, S, sl2, ws, nullptr, AppendState{});
    else
      decode_split_kernel<T, 64, false><<<grid, block, 0, s>>>(
          static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), key_len,
          H, Nk, S, sl2, ws, nullptr, AppendState{});
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_merge<true>(ws.m, ws.l, ws.o, S, rows, d, dt, o, lse, s);
}

// ---------------------------------------------------------------------------
// Allocation-free decode.  Callers that cannot allocate device memory get the
// split summaries kept in this fixed-size device array instead of a workspace
// of their own.  Host code must not hand the array's name to a kernel (on the
// host it is only a stand-in symbol, not a device address): the device
// address is looked up with cudaGetSymbolAddress once per device and context
// and cached together with the context's unique id, so a new context on the
// device (after cudaDeviceReset, say) is seen and the address looked up again.
namespace {
static __device__ __align__(256) unsigned char g_noalloc_scratch[OSM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxCachedDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxCachedDevices] = {};
unsigned long long g_noalloc_ctx[kMaxCachedDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The unique id of the calling thread's current context (0 if unknown).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

cudaError_t noalloc_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cacheable = dev >= 0 && dev < kMaxCachedDevices;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  const unsigned long long ctx = current_context_id();
  if (cacheable && ctx != 0 && g_noalloc_ptr[dev] != nullptr && g_noalloc_ctx[dev] == ctx) {
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // the current device's copy
  if (e != cudaSuccess) return e;
  if (cacheable) {
    g_noalloc_ptr[dev] = p;
    g_noalloc_ctx[dev] = current_context_id();  // the context now exists
  }
  *out = p;
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_decode_splitkv_noalloc(osm_dtype dt, const void* q, const void* k,
                                          const void* v, void* o, float* lse, int B, int H,
                                          int Nk, int d, float scale, const int32_t* key_len,
                                          int S, cudaStream_t s) {
  void* scratch = nullptr;
  cudaError_t e = noalloc_scratch_address(&scratch);
  if (e != cudaSuccess) return e;
  return launch_decode_splitkv(dt, q, k, v, o, lse, B, H, Nk, d, scale, key_len, S, scratch, s);
}

cudaError_t read_and_clear_decode_check(uint32_t* word) {
  unsigned int w = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&w, g_chk_word, sizeof(w));
  if (e != cudaSuccess) return e;
  if (w != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_chk_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
  }
  *word = w;
  return cudaSuccess;
}

size_t decode_append_workspace_bytes(int B, int H, int d, int S) {
  return decode_workspace_bytes(B, H, d, S) + ws_section(static_cast<int64_t>(B) * H);
}

cudaError_t launch_decode_append(osm_dtype dt, const void* q, const void* k, const void* v,
                                 int B, int H, int Nk, int d, float scale,
                                 const int32_t* key_start, const int32_t* key_end, float* state_m,
                                 float* state_l, float* state_o, void* o, float* lse, int S,
                                 void* ws_ptr, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(B) * H;
  Workspace ws = carve(ws_ptr, rows * S, d);
  unsigned int* tickets = reinterpret_cast<unsigned int*>(
      static_cast<char*>(ws_ptr) + decode_workspace_bytes(B, H, d, S));
  cudaError_t e = cudaMemsetAsync(tickets, 0, static_cast<size_t>(rows) * 4, s);
  if (e != cudaSuccess) return e;
  const AppendState st{state_m, state_l, state_o, o, lse, dt == OSM_BF16 ? 1 : 0, tickets};
  const float sl2 = scale * kLog2e;
  const dim3 grid(S, H, B), block(kWarps * 32);
  if (dt == OSM_BF16) {
    using T = __nv_bfloat16;
    const T *tq = static_cast<const T*>(q), *tk = static_cast<const T*>(k),
            *tv = static_cast<const T*>(v);
    if (d == 128)
      decode_split_kernel<T, 128, true>
          <<<grid, block, 0, s>>>(tq, tk, tv, key_end, H, Nk, S, sl2, ws, key_start, st);
    else
      decode_split_kernel<T, 64, true>
          <<<grid, block, 0, s>>>(tq, tk, tv, key_end, H, Nk, S, sl2, ws, key_start, st);
  } else {
    using T = float;
    const T *tq = static_cast<const T*>(q), *tk = static_cast<const T*>(k),
            *tv = static_cast<const T*>(v);
    if (d == 128)
      decode_split_kernel<T, 128, true>
          <<<grid, block, 0, s>>>(tq, tk, tv, key_end, H, Nk, S, sl2, ws, key_start, st);
    else
      decode_split_kernel<T, 64, true>
          <<<grid, block, 0, s>>>(tq, tk, tv, key_end, H, Nk, S, sl2, ws, key_start, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(const float* o_parts, const float* lse_parts, int S, int64_t rows,
                             int d, osm_dtype out_dt, void* o, float* lse, cudaStream_t s) {
  return launch_merge<false>(lse_parts, nullptr, o_parts, S, rows, d, out_dt, o, lse, s);
}

}  // namespace osm
