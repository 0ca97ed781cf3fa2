// softmax_rows.cu — FP32 row softmax with the online normaliser.
//
// "Online softmax" (zerotofrontier.app), sections "The recurrence, and a proof
// that it is right" and "Merging partial results": a row is cut into pieces,
// each piece is summarised as (m, l) = (max, sum of exp(x - max)), and the
// summaries are merged exactly in any grouping — here a warp-shuffle tree, then
// across the warps of a CTA, then across the CTAs of a thread-block cluster
// through distributed shared memory: each CTA sends its summary to every CTA
// of the cluster with an asynchronous store that completes bytes on the
// receiver's mbarrier, so a CTA waits only for the summaries it needs (no
// cluster-wide barrier after the exchange; 5.90 -> 6.39 TB/s on 4096 x
// 32768).  Every CTA merges the cluster's summaries in the same rank order,
// so all of them hold the same (M, L); each then writes y = exp(x - M) / L
// for its piece.
//
// Fast path: the row stays in registers between the summary and the scaling
// pass, so x is read from HBM once and y written once (8 bytes per element,
// below the 3 accesses per element of the pages' two-pass form).  Fallback
// (unaligned rows or rows over 131072 columns): the pages' two-pass form,
// x read twice.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "exp_le0.cuh"
#include "ptx.cuh"

namespace osm {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();

// weight of a summary with max m when brought to the common max mn (mn >= m);
// an empty summary (m = -inf) weighs 0.
__device__ __forceinline__ float rebase(float m, float mn) {
  return m == kNegInf ? 0.f : ptx::ex2((m - mn) * kLog2e);
}

// merge (m, l) with (mo, lo) in place
__device__ __forceinline__ void merge_ml(float& m, float& l, float mo, float lo) {
  const float mn = fmaxf(m, mo);
  l = l * rebase(m, mn) + lo * rebase(mo, mn);
  m = mn;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// error word of the row-softmax kernels: a summary wait that ran out
__device__ unsigned int g_softmax_err;
constexpr unsigned kSoftmaxSite = 0x03000001u;

// 8 bytes into the shared memory of CTA `rank` of this cluster (at the address
// `local` has in this CTA), completing that many bytes on the mbarrier at
// `local_bar`'s address in that CTA
__device__ __forceinline__ void st_async_f2(const void* local, const void* local_bar, uint32_t rank,
                                            float a, float b) {
  uint32_t ra, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(ptx::smem_u32(local)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(ptx::smem_u32(local_bar)), "r"(rank));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
               ::"r"(ra), "f"(a), "f"(b), "r"(rb)
               : "memory");
}

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;

// One cluster of `nct` CTAs per row; CTA `rank` owns float4 columns
// [rank*kThreads*V, (rank+1)*kThreads*V) of the row, V per thread.
template <int V>
__global__ void __launch_bounds__(kThreads, 5) softmax_rows_cluster(const float* __restrict__ x,
                                                                  float* __restrict__ y,
                                                                  int cols) {
  __shared__ float2 warp_ml[kWarps];
  __shared__ __align__(8) float2 cta_ml[kMaxCluster];
  __shared__ __align__(8) uint64_t ml_bar;  // completes when every CTA's summary has arrived
  __shared__ int abort_flag;

  const uint32_t nct = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const int64_t row = blockIdx.x / nct;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cols4 = cols >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x + row * static_cast<int64_t>(cols));
  float4* yr = reinterpret_cast<float4*>(y + row * static_cast<int64_t>(cols));
  const int base4 = static_cast<int>(rank) * kThreads * V + tid;

  // the summary barrier is set up (expecting nct summaries of 8 bytes) before
  // the cluster barrier, so no peer writes before it exists
  if (threadIdx.x == 0) {
    abort_flag = 0;
    ptx::mbar_init(ptx::smem_u32(&ml_bar), 1);
    ptx::fence_mbar_init();
    ptx::mbar_arrive_expect_tx(ptx::smem_u32(&ml_bar), 8u * nct);
  }
  __syncthreads();
  cluster_arrive_release();

  float4 v[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int c4 = base4 + i * kThreads;
    v[i] = c4 < cols4 ? __ldcs(xr + c4) : make_float4(kNegInf, kNegInf, kNegInf, kNegInf);
  }

  // this thread's summary: max, then sum of exp(x - max)
  float m = kNegInf;
#pragma unroll
  for (int i = 0; i < V; ++i) m = fmaxf(m, fmaxf(fmaxf(v[i].x, v[i].y), fmaxf(v[i].z, v[i].w)));
  // (x - m) first: exact near the max whatever the magnitude of m
  float l = 0.f;
  if (m != kNegInf) {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      l += ptx::ex2((v[i].x - m) * kLog2e) + ptx::ex2((v[i].y - m) * kLog2e) +
           ptx::ex2((v[i].z - m) * kLog2e) + ptx::ex2((v[i].w - m) * kLog2e);
    }
  }
  // warp tree
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off);
    const float lo = __shfl_xor_sync(0xffffffffu, l, off);
    merge_ml(m, l, mo, lo);
  }
  if (lane == 0) warp_ml[warp] = make_float2(m, l);
  __syncthreads();
  // CTA summary, merged in warp order
  float mc = warp_ml[0].x, lc = warp_ml[0].y;
#pragma unroll
  for (int w = 1; w < kWarps; ++w) merge_ml(mc, lc, warp_ml[w].x, warp_ml[w].y);

  cluster_wait_acquire();  // every CTA of the cluster has set up its barrier
  if (tid < static_cast<int>(nct)) st_async_f2(&cta_ml[rank], &ml_bar, tid, mc, lc);
  // a wait that runs out records the error and goes on with what has arrived
  ptx::wait_bounded(ptx::smem_u32(&ml_bar), 0, &abort_flag, &g_softmax_err, kSoftmaxSite);

  // row summary, merged in rank order (identical in every CTA of the cluster)
  float M = cta_ml[0].x, L = cta_ml[0].y;
  for (uint32_t r = 1; r < nct; ++r) merge_ml(M, L, cta_ml[r].x, cta_ml[r].y);
  const float inv = L > 0.f ? 1.f / L : 0.f;

#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int c4 = base4 + i * kThreads;
    if (c4 < cols4) {
      float4 o;
      o.x = exp_le0(v[i].x - M) * inv;
      o.y = exp_le0(v[i].y - M) * inv;
      o.z = exp_le0(v[i].z - M) * inv;
      o.w = exp_le0(v[i].w - M) * inv;
      __stcs(yr + c4, o);
    }
  }
}

// Generic two-pass kernel, one CTA per row, any alignment and length.
// Pass 1: each thread runs the running (max, sum) recurrence over its strided
// elements, four at a time; the summaries are merged across the CTA.  Pass 2
// re-reads x and writes y = exp(x - M) / L.
constexpr int kGenThreads = 512;
__global__ void __launch_bounds__(kGenThreads) softmax_rows_generic(const float* x, float* y,
                                                                    int64_t cols) {
  __shared__ float2 warp_ml[kGenThreads / 32];
  const int64_t row = blockIdx.x;
  const float* xr = x + row * cols;
  float* yr = y + row * cols;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float m = kNegInf, l = 0.f;
  for (int64_t c = tid; c < cols; c += 4 * kGenThreads) {
    float a[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t cc = c + u * kGenThreads;
      a[u] = cc < cols ? xr[cc] : kNegInf;
    }
    const float mt = fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3]));
    if (mt == kNegInf) continue;
    const float mn = fmaxf(m, mt);
    float s = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) s += ptx::ex2((a[u] - mn) * kLog2e);
    l = l * rebase(m, mn) + s;
    m = mn;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off);
    const float lo = __shfl_xor_sync(0xffffffffu, l, off);
    merge_ml(m, l, mo, lo);
  }
  if (lane == 0) warp_ml[warp] = make_float2(m, l);
  __syncthreads();
  float M = warp_ml[0].x, L = warp_ml[0].y;
  for (int w = 1; w < kGenThreads / 32; ++w) merge_ml(M, L, warp_ml[w].x, warp_ml[w].y);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  for (int64_t c = tid; c < cols; c += kGenThreads) yr[c] = exp_le0(xr[c] - M) * inv;
}

template <int V>
cudaError_t launch_cluster(const float* x, float* y, int64_t rows, int cols, int nct,
                           cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(rows * nct), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nct;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, softmax_rows_cluster<V>, x, y, cols);
}

}  // namespace

cudaError_t launch_softmax_rows(const float* x, float* y, int64_t rows, int64_t cols,
                                cudaStream_t s) {
  const bool aligned = (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(y) % 16 == 0) && (cols % 4 == 0);
  if (aligned && cols <= 131072) {
    // columns per CTA = kThreads * 4 * V; one CTA per row while 8 float4 per
    // thread cover it, else clusters of 8-float4 slices (16 past 8 CTAs)
    int V = 16;
    for (int cand : {2, 4, 8}) {
      if (cols <= kThreads * 4 * cand) {
        V = cand;
        break;
      }
    }
    if (V == 16 && (cols + kThreads * 32 - 1) / (kThreads * 32) <= 8) V = 8;
    const int per = kThreads * 4 * V;
    const int nct = static_cast<int>((cols + per - 1) / per);
    if (rows * nct <= 0x7fffffffLL) {
      switch (V) {
        case 2: return launch_cluster<2>(x, y, rows, static_cast<int>(cols), nct, s);
        case 4: return launch_cluster<4>(x, y, rows, static_cast<int>(cols), nct, s);
        case 8: return launch_cluster<8>(x, y, rows, static_cast<int>(cols), nct, s);
        default: return launch_cluster<16>(x, y, rows, static_cast<int>(cols), nct, s);
      }
    }
  }
  softmax_rows_generic<<<static_cast<unsigned>(rows), kGenThreads, 0, s>>>(x, y, cols);
  return cudaGetLastError();
}

cudaError_t read_and_clear_softmax_error(uint32_t* word) {
  unsigned int w = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&w, g_softmax_err, sizeof(w));
  if (e != cudaSuccess) return e;
  if (w != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_softmax_err, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
  }
  *word = w;
  return cudaSuccess;
}

}  // namespace osm
