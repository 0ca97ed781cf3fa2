// softmax_topk.cu — fused online softmax + top-k of every row, one read of x.
//
// "Online softmax" (zerotofrontier.app), the `softmax_topk` exercise after
// "Precision, and what can still go wrong", and the reading list's Milakov &
// Gimelshein entry: the indices of a row's k largest scores together with
// their softmax probabilities, from one pass over the row.  Each thread keeps
// the online normaliser (m, l) of its elements ("The recurrence, and a proof
// that it is right") and a sorted list of its k best (value, index) pairs;
// both kinds of summary merge exactly in any grouping ("Merging partial
// results"), so the row's result is assembled warp -> CTA -> thread-block
// cluster.  Order: larger value first, equal values by smaller index, so the
// result is unique.  Probabilities are exp(x_i - M) / L with the row's (M, L).
//
// GB300 mapping: one cluster of nct CTAs (256 threads each) per row; CTA r of
// the cluster streams a contiguous slice of the row with 16-byte loads, four
// in flight per thread.  Lists merge by k rounds of a warp-wide arg-max over
// the lanes' list heads; the CTA's lists meet in shared memory and the
// cluster's in CTA 0 through distributed shared memory.  HBM-bound: 4 bytes
// read per element, 8 bytes written per output entry.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace osm {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;
// log2(e) split into an fp32 head and its remainder, for argument reduction
constexpr float kLog2eHi = 1.44269502162933349609375f;
constexpr float kLog2eLo = 1.925963033500011079e-8f;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr int kNoIndex = 0x7fffffff;  // empty list slot: after every real entry

// the total order of (value, index) pairs
__device__ __forceinline__ bool before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// exp(d) for d <= 0 (Cody & Waite split of d*log2(e) into an integer and a
// remainder, so the remainder keeps full precision); flushes below 2^-125
__device__ __forceinline__ float exp_le0(float d) {
  d = fmaxf(d, -100.f);
  const float n = rintf(d * kLog2eHi);
  float f = fmaf(d, kLog2eHi, -n);
  f = fmaf(d, kLog2eLo, f);
  const float r = ptx::ex2(f);
  const int ni = static_cast<int>(n);
  return ni < -125 ? 0.f : r * __int_as_float((ni + 127) << 23);
}

// K best (value, index) pairs seen so far, sorted by the order above
template <int K>
struct List {
  float v[K];
  int i[K];
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int s = 0; s < K; ++s) {
      v[s] = kNegInf;
      i[s] = kNoIndex;
    }
  }
  __device__ __forceinline__ void insert(float x, int j) {
    if (!before(x, j, v[K - 1], i[K - 1])) return;
#pragma unroll
    for (int s = K - 1; s >= 0; --s) {  // reads v[s], v[s-1] before either is written
      if (s > 0 && before(x, j, v[s - 1], i[s - 1])) {
        v[s] = v[s - 1];
        i[s] = i[s - 1];
      } else if (before(x, j, v[s], i[s])) {
        v[s] = x;
        i[s] = j;
      }
    }
  }
  __device__ __forceinline__ void pop() {
#pragma unroll
    for (int s = 0; s + 1 < K; ++s) {
      v[s] = v[s + 1];
      i[s] = i[s + 1];
    }
    v[K - 1] = kNegInf;
    i[K - 1] = kNoIndex;
  }
};

// The K best entries over the lists of all lanes of the warp, by K rounds of a
// warp-wide arg-max over the list heads.  Rank r ends in lane r % 32 (slot 0
// for r < 32, slot 1 for 32 <= r < 64).
template <int K>
__device__ __forceinline__ void warp_merge(List<K>& L, float& v0, int& i0, float& v1, int& i1) {
  const int lane = threadIdx.x & 31;
  v0 = v1 = kNegInf;
  i0 = i1 = kNoIndex;
#pragma unroll 1
  for (int r = 0; r < K; ++r) {
    float bv = L.v[0];
    int bi = L.i[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (before(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi != kNoIndex && L.i[0] == bi) L.pop();  // indices are unique within a row
    if ((r & 31) == lane) {
      if (r < 32) {
        v0 = bv;
        i0 = bi;
      } else {
        v1 = bv;
        i1 = bi;
      }
    }
  }
}

__device__ __forceinline__ float rebase(float m, float mn) {  // weight of a summary at max mn
  return m == kNegInf ? 0.f : ptx::ex2((m - mn) * kLog2e);
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_addr(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(ptx::smem_u32(local)), "r"(rank));
  return remote;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

template <int K>
struct Block {  // per (value, index) pair feeding: online (m, l) and the list
  float m = kNegInf, l = 0.f;
  List<K> L;
  __device__ __forceinline__ void add4(float4 x, int j) {
    const float mb = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
    if (mb > m) {
      l = (m == kNegInf) ? 0.f : l * ptx::ex2((m - mb) * kLog2e);
      m = mb;
    }
    if (m != kNegInf)
      l += (ptx::ex2((x.x - m) * kLog2e) + ptx::ex2((x.y - m) * kLog2e)) +
           (ptx::ex2((x.z - m) * kLog2e) + ptx::ex2((x.w - m) * kLog2e));
    L.insert(x.x, j);
    L.insert(x.y, j + 1);
    L.insert(x.z, j + 2);
    L.insert(x.w, j + 3);
  }
  __device__ __forceinline__ void add1(float x, int j) {
    if (x > m) {
      l = (m == kNegInf) ? 0.f : l * ptx::ex2((m - x) * kLog2e);
      m = x;
    }
    if (m != kNegInf) l += ptx::ex2((x - m) * kLog2e);
    L.insert(x, j);
  }
};

template <int K>
__global__ void __launch_bounds__(kThreads) softmax_topk_kernel(const float* __restrict__ x,
                                                                int64_t cols, int nct, int vec,
                                                                int k, int32_t* __restrict__ idx,
                                                                float* __restrict__ prob) {
  __shared__ float s_v[kWarps][K];
  __shared__ int s_i[kWarps][K];
  __shared__ float s_m[kWarps], s_l[kWarps];
  __shared__ float c_v[K];  // this CTA's list and summary, read by CTA 0 of the cluster
  __shared__ int c_i[K];
  __shared__ float c_ml[2];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int64_t row = blockIdx.x / nct;
  const float* xr = x + row * cols;
  // this CTA's slice of the row (a multiple of 4 columns long)
  const int64_t chunk = ((cols + nct - 1) / nct + 3) / 4 * 4;
  const int64_t c0 = rank * chunk < cols ? rank * chunk : cols;
  const int64_t c1 = c0 + chunk < cols ? c0 + chunk : cols;

  Block<K> st;
  st.L.clear();
  if (vec) {
    const float4* x4 = reinterpret_cast<const float4*>(xr);
    const int64_t f0 = c0 / 4, f1 = c1 / 4;
    int64_t f = f0 + tid;
    for (; f + 3 * kThreads < f1; f += 4 * kThreads) {  // four 16-byte loads in flight
      const float4 a = __ldcs(x4 + f), b = __ldcs(x4 + f + kThreads);
      const float4 c = __ldcs(x4 + f + 2 * kThreads), d = __ldcs(x4 + f + 3 * kThreads);
      st.add4(a, static_cast<int>(4 * f));
      st.add4(b, static_cast<int>(4 * (f + kThreads)));
      st.add4(c, static_cast<int>(4 * (f + 2 * kThreads)));
      st.add4(d, static_cast<int>(4 * (f + 3 * kThreads)));
    }
    for (; f < f1; f += kThreads) st.add4(__ldcs(x4 + f), static_cast<int>(4 * f));
  } else {
    for (int64_t j = c0 + tid; j < c1; j += kThreads) st.add1(__ldcs(xr + j), static_cast<int>(j));
  }

  // warp: (m, l) by shuffles, lists by K rounds
  float m = st.m, l = st.l;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off);
    const float lo = __shfl_xor_sync(0xffffffffu, l, off);
    const float mn = fmaxf(m, mo);
    l = l * rebase(m, mn) + lo * rebase(mo, mn);
    m = mn;
  }
  float v0, v1;
  int i0, i1;
  warp_merge<K>(st.L, v0, i0, v1, i1);
  if (lane < K) {
    s_v[warp][lane] = v0;
    s_i[warp][lane] = i0;
  }
  if (lane + 32 < K) {
    s_v[warp][lane + 32] = v1;
    s_i[warp][lane + 32] = i1;
  }
  if (lane == 0) {
    s_m[warp] = m;
    s_l[warp] = l;
  }
  __syncthreads();
  // CTA: warp 0 merges the warps' lists (lane w holds warp w's list)
  if (warp == 0) {
    List<K> L;
    L.clear();
    if (lane < kWarps) {
#pragma unroll
      for (int s = 0; s < K; ++s) {
        L.v[s] = s_v[lane][s];
        L.i[s] = s_i[lane][s];
      }
    }
    warp_merge<K>(L, v0, i0, v1, i1);
    if (lane < K) {
      c_v[lane] = v0;
      c_i[lane] = i0;
    }
    if (lane + 32 < K) {
      c_v[lane + 32] = v1;
      c_i[lane + 32] = i1;
    }
    if (lane == 0) {
      float M = s_m[0], Ls = s_l[0];
      for (int w = 1; w < kWarps; ++w) {
        const float mn = fmaxf(M, s_m[w]);
        Ls = Ls * rebase(M, mn) + s_l[w] * rebase(s_m[w], mn);
        M = mn;
      }
      c_ml[0] = M;
      c_ml[1] = Ls;
    }
  }
  cluster_sync_all();  // every CTA's list and summary are visible to CTA 0
  if (rank == 0 && warp == 0) {
    List<K> L;
    L.clear();
    if (lane < nct) {
#pragma unroll
      for (int s = 0; s < K; ++s) {
        L.v[s] = ld_cluster_f32(cluster_addr(&c_v[s], lane));
        L.i[s] = ld_cluster_s32(cluster_addr(&c_i[s], lane));
      }
    }
    warp_merge<K>(L, v0, i0, v1, i1);
    // the row's (M, L), merged in rank order
    float M = kNegInf, Ls = 0.f;
    for (int q = 0; q < nct; ++q) {
      const float mq = ld_cluster_f32(cluster_addr(&c_ml[0], q));
      const float lq = ld_cluster_f32(cluster_addr(&c_ml[1], q));
      const float mn = fmaxf(M, mq);
      Ls = Ls * rebase(M, mn) + lq * rebase(mq, mn);
      M = mn;
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    int32_t* irow = idx + row * k;
    float* prow = prob + row * k;
    if (lane < k) {
      irow[lane] = i0;
      prow[lane] = (Ls > 0.f && v0 != kNegInf) ? exp_le0(v0 - M) * inv : 0.f;
    }
    if (lane + 32 < k) {
      irow[lane + 32] = i1;
      prow[lane + 32] = (Ls > 0.f && v1 != kNegInf) ? exp_le0(v1 - M) * inv : 0.f;
    }
  }
  cluster_sync_all();  // CTA 0 has read every CTA's shared memory
}

template <int K>
cudaError_t launch_k(const float* x, int64_t rows, int64_t cols, int k, int nct, int vec,
                     int32_t* idx, float* prob, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(rows * nct));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nct;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, softmax_topk_kernel<K>, x, cols, nct, vec, k, idx, prob);
}

}  // namespace

cudaError_t launch_softmax_topk(const float* x, int64_t rows, int64_t cols, int k, int32_t* idx,
                                float* prob, cudaStream_t s) {
  const int vec = (cols % 4 == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0) ? 1 : 0;
  // enough CTAs to cover the SMs a few times over; every CTA keeps >= 8192 columns
  const int64_t want = 4LL * sm_count_current_device();
  int nct = 1;
  while (nct < 8 && rows * nct < want && cols / (2 * nct) >= 8192) nct *= 2;
  if (k <= 1) return launch_k<1>(x, rows, cols, k, nct, vec, idx, prob, s);
  if (k <= 2) return launch_k<2>(x, rows, cols, k, nct, vec, idx, prob, s);
  if (k <= 4) return launch_k<4>(x, rows, cols, k, nct, vec, idx, prob, s);
  if (k <= 8) return launch_k<8>(x, rows, cols, k, nct, vec, idx, prob, s);
  if (k <= 16) return launch_k<16>(x, rows, cols, k, nct, vec, idx, prob, s);
  return launch_k<32>(x, rows, cols, k, nct, vec, idx, prob, s);
}

}  // namespace osm
