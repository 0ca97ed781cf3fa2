// softmax_topk.cu — fused online softmax + top-k of every row; x comes from
// HBM once.
//
// "Online softmax" (zerotofrontier.app), the `softmax_topk` exercise after
// "Precision, and what can still go wrong", and the reading list's Milakov &
// Gimelshein entry: the indices of a row's k largest scores together with
// their softmax probabilities, fused with the normaliser.  Threads keep the
// online normaliser (m, l) of their elements ("The recurrence, and a proof
// that it is right") and warps keep sorted lists of their best (value, index)
// pairs; both kinds of summary merge exactly in any grouping ("Merging
// partial results"), so the row's result is assembled warp -> CTA ->
// thread-block cluster.  Order: larger value first, equal values by smaller
// index, so the result is unique.  Probabilities are exp(x_i - M) / L with
// the row's (M, L).
//
// GB300 mapping: one cluster of nct CTAs (256 threads each) per row; CTA r of
// the cluster streams a contiguous slice of the row with 16-byte loads, four
// in flight per thread.  That pass forms (m, l), each thread's maximum and
// the maximum of each of its groups of 16 entries (kept in shared memory);
// the k-th largest thread maximum within the warp (within the CTA for
// k > 16) is a threshold every top-k entry reaches.  Only the groups whose
// maximum reaches it are read again (from L2, mostly): the warp shares them
// out one per lane, and the entries that beat the warp's filter enter the
// warp's running list of 32 pairs, one per lane, by insertion when a round
// offers few and by a sort and merge when it offers many; the filter tightens
// to the list's k-th entry.  The CTA's lists meet pairwise through shared
// memory (three rounds for eight warps) and the cluster's in CTA 0 through
// distributed shared memory, by bitonic merges.  K = 1 needs one pass (each
// thread's arg-max).  HBM-bound: 4 bytes read per element once from HBM (plus
// the few groups read again), 8 bytes written per output entry.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "exp_le0.cuh"
#include "ptx.cuh"

namespace osm {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kMaxFloat = 3.402823466e38f;
constexpr int kNoIndex = 0x7fffffff;  // empty list slot: after every real entry
// K > 1: the maxima of a thread's groups of 16 entries (the four 16-byte
// loads of one step of the first pass) kept for the second pass; groups past
// kGroupSlots share slot g mod kGroupSlots (kept as the maximum over them)
constexpr int kGroupSlots = 16;

// the total order of (value, index) pairs
__device__ __forceinline__ bool before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// position of the n-th (0-based) set bit of m; n < popc(m)
__device__ __forceinline__ int nth_set_bit(unsigned m, int n) {
  int pos = 0;
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) {
    const int c = __popc(m & ((1u << w) - 1u));
    if (n >= c) {
      n -= c;
      m >>= w;
      pos += w;
    }
  }
  return pos;
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

// Lane-sorted lists of (value, index) pairs: lane r holds the r-th entry in
// the total order above.  Compare-exchange with the partner lane^stride, keeping
// the better entry when keep_best.
__device__ __forceinline__ void cmpx_pair(float& v, int& i, int stride, bool keep_best) {
  const float ov = __shfl_xor_sync(0xffffffffu, v, stride);
  const int oi = __shfl_xor_sync(0xffffffffu, i, stride);
  if (before(ov, oi, v, i) == keep_best) {
    v = ov;
    i = oi;
  }
}
// One pair per lane -> the warp's 32 pairs sorted (bitonic network, 15 stages).
__device__ __forceinline__ void warp_sort_pairs(float& v, int& i) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size / 2; stride > 0; stride >>= 1)
      cmpx_pair(v, i, stride, ((lane & stride) == 0) == ((lane & size) == 0));
  }
}
// a <- the 32 best of the lane-sorted lists a and b, lane-sorted.
__device__ __forceinline__ void warp_merge_pairs(float& av, int& ai, float bv, int bi) {
  const int lane = threadIdx.x & 31;
  const float rv = __shfl_sync(0xffffffffu, bv, 31 - lane);
  const int ri = __shfl_sync(0xffffffffu, bi, 31 - lane);
  if (!before(av, ai, rv, ri)) {  // the better of a[r] and b[31-r]: a bitonic sequence
    av = rv;
    ai = ri;
  }
#pragma unroll
  for (int stride = 16; stride > 0; stride >>= 1) cmpx_pair(av, ai, stride, (lane & stride) == 0);
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
// a cluster barrier when the row spans several CTAs, else the CTA's own
// (cheaper; nct is the same in every thread)
__device__ __forceinline__ void row_sync(int nct) {
  if (nct > 1) cluster_sync_all();
  else __syncthreads();
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

// One value per lane -> the warp's 32 values sorted in descending order
// (lane r holds the r-th largest): a bitonic network of 15 shuffle stages.
__device__ __forceinline__ float warp_sort_desc(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size / 2; stride > 0; stride >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
      v = keep_max ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return v;
}
// The 32 largest of two descending lane-sorted lists, again lane-sorted.
__device__ __forceinline__ float warp_merge_desc(float a, float b) {
  const int lane = threadIdx.x & 31;
  float c = fmaxf(a, __shfl_sync(0xffffffffu, b, 31 - lane));  // bitonic, holds the top 32
#pragma unroll
  for (int stride = 16; stride > 0; stride >>= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, c, stride);
    c = (lane & stride) == 0 ? fmaxf(c, o) : fminf(c, o);
  }
  return c;
}


// The CTA's warps' lane-sorted lists (s_pv/s_pi, 32 per warp) merged pairwise
// in log2(kWarps) rounds; the result ends in warp 0's entries.  Every thread
// of the CTA calls this (it holds the barriers).
__device__ __forceinline__ void cta_tree_merge_pairs(float* s_pv, int* s_pi) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int step = 1; step < kWarps; step <<= 1) {
    __syncthreads();
    if ((warp & (2 * step - 1)) == 0) {
      float av = s_pv[warp * 32 + lane];
      int ai = s_pi[warp * 32 + lane];
      warp_merge_pairs(av, ai, s_pv[(warp + step) * 32 + lane], s_pi[(warp + step) * 32 + lane]);
      __syncwarp();
      s_pv[warp * 32 + lane] = av;
      s_pi[warp * 32 + lane] = ai;
    }
  }
  __syncthreads();
}

// The 32 best entries over the per-thread lists of a whole cluster, lane-sorted
// in warp 0 of CTA 0.  Warp: the lanes' r-th entries are sorted as a batch and
// merged into the running list, one batch per list depth in use; CTA: warp 0
// merges the warps' lists from shared memory; cluster: CTA 0's warp 0 merges
// the CTAs' lists through distributed shared memory.  One cluster barrier
// inside; the caller adds another before the shared lists are written again.
template <int K>
__device__ __forceinline__ void cluster_topk(List<K>& L, float* s_pv, int* s_pi,
                                             float* c_v, int* c_i, int nct, uint32_t rank,
                                             float& av, int& ai) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  av = kNegInf;
  ai = kNoIndex;
#pragma unroll 1
  for (int r = 0; r < K; ++r) {
    if (!__any_sync(0xffffffffu, L.i[0] != kNoIndex)) break;  // lists are filled in order
    float bv = L.v[0];
    int bi = L.i[0];
    L.pop();
    warp_sort_pairs(bv, bi);
    if (r == 0) {
      av = bv;
      ai = bi;
    } else {
      warp_merge_pairs(av, ai, bv, bi);
    }
  }
  s_pv[warp * 32 + lane] = av;
  s_pi[warp * 32 + lane] = ai;
  cta_tree_merge_pairs(s_pv, s_pi);
  if (warp == 0) {
    av = s_pv[lane];
    ai = s_pi[lane];
    c_v[lane] = av;
    c_i[lane] = ai;
  }
  row_sync(nct);  // every CTA's list is visible to CTA 0
  if (rank == 0 && warp == 0) {
    for (int q = 1; q < nct; ++q)
      warp_merge_pairs(av, ai, ld_cluster_f32(cluster_addr(&c_v[lane], q)),
                       ld_cluster_s32(cluster_addr(&c_i[lane], q)));
  }
}

// The 32 best entries of the cluster from each warp's lane-sorted list (av, ai),
// lane-sorted in warp 0 of CTA 0; as the tail of cluster_topk.
// Also merges the warps' (m, l) (s_m, s_l) into the CTA's (c_ml).
__device__ __forceinline__ void cluster_merge_lists(float& av, int& ai, float* s_pv, int* s_pi,
                                                    const float* s_m, const float* s_l,
                                                    float* c_ml, float* c_v, int* c_i, int nct,
                                                    uint32_t rank) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  s_pv[warp * 32 + lane] = av;
  s_pi[warp * 32 + lane] = ai;
  cta_tree_merge_pairs(s_pv, s_pi);
  if (threadIdx.x == 32) {  // the CTA's (m, l), read by CTA 0 at the end
    float M = s_m[0], Ls = s_l[0];
    for (int w = 1; w < kWarps; ++w) {
      const float mn = fmaxf(M, s_m[w]);
      Ls = Ls * rebase(M, mn) + s_l[w] * rebase(s_m[w], mn);
      M = mn;
    }
    c_ml[0] = M;
    c_ml[1] = Ls;
  }
  if (warp == 0) {
    av = s_pv[lane];
    ai = s_pi[lane];
    c_v[lane] = av;
    c_i[lane] = ai;
  }
  row_sync(nct);  // every CTA's list is visible to CTA 0
  if (rank == 0 && warp == 0) {
    for (int q = 1; q < nct; ++q)
      warp_merge_pairs(av, ai, ld_cluster_f32(cluster_addr(&c_v[lane], q)),
                       ld_cluster_s32(cluster_addr(&c_i[lane], q)));
  }
}

// Two passes over the CTA's slice of the row (the second over a few groups):
//  1. the online (m, l), each thread's maximum and its groups' maxima; the
//     K-th largest thread maximum of a warp is a threshold T with at least K
//     entries of the warp >= T, so every entry of the row's top K is >= its
//     warp's T, and lies in a group whose maximum is >= T;
//  2. only entries of those groups that beat the warp's filter (T, then the
//     K-th entry of the warp's running list) enter that list; the warps'
//     lists merge into the row's top K.  K = 1 needs one pass: each thread's
//     argmax.
// (registers capped for six CTAs per SM, eight for the one-pass K = 1)
template <int K>
__global__ void __launch_bounds__(kThreads, K > 1 ? 6 : 8)
    softmax_topk_kernel(const float* __restrict__ x, int64_t cols, int nct, int vec, int k,
                        int32_t* __restrict__ idx, float* __restrict__ prob) {
  __shared__ float s_pv[kWarps * 32];  // the warps' sorted lists
  __shared__ int s_pi[kWarps * 32];
  __shared__ float s_m[kWarps], s_l[kWarps];
  __shared__ float c_v[32];  // this CTA's list and summary, read by CTA 0 of the cluster
  __shared__ int c_i[32];
  __shared__ float c_ml[2];
  __shared__ float s_gm[(K > 1 ? kGroupSlots : 1) * kThreads];  // K > 1: the group maxima

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int64_t row = blockIdx.x / nct;
  const float* xr = x + row * cols;
  // this CTA's slice of the row (a multiple of 4 columns long)
  const int64_t chunk = ((cols + nct - 1) / nct + 3) / 4 * 4;
  const int64_t c0 = rank * chunk < cols ? rank * chunk : cols;
  const int64_t c1 = c0 + chunk < cols ? c0 + chunk : cols;
  const float4* x4 = reinterpret_cast<const float4*>(xr);
  const int64_t f0 = c0 / 4, f1 = c1 / 4;

  // ---- pass 1: (m, l) and the thread maximum.  m starts at the lowest
  // finite float rather than -inf, so the updates need no branch: a group of
  // -inf entries adds exp2(-inf) = 0 and rescales by exp2(0) = 1.
  float m = -kMaxFloat, l = 0.f;
  float bv = kNegInf;  // K == 1: the thread's best entry (elements arrive in column order)
  int bi = kNoIndex;
  auto best = [&](float v, int j) {
    if constexpr (K == 1) {
      const bool t = v > bv || bi == kNoIndex;
      bv = t ? v : bv;
      bi = t ? j : bi;
    }
  };
  auto add1 = [&](float v) {
    if (v > m) {
      l = (m == kNegInf) ? 0.f : l * ptx::ex2((m - v) * kLog2e);
      m = v;
    }
    if (m != kNegInf) l += ptx::ex2((v - m) * kLog2e);
  };
  auto add4 = [&](float4 v) {
    const float mb = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
    if (mb > m) {
      l = (m == kNegInf) ? 0.f : l * ptx::ex2((m - mb) * kLog2e);
      m = mb;
    }
    if (m != kNegInf)
      l += (ptx::ex2((v.x - m) * kLog2e) + ptx::ex2((v.y - m) * kLog2e)) +
           (ptx::ex2((v.z - m) * kLog2e) + ptx::ex2((v.w - m) * kLog2e));
  };
  // group g of this thread: float4s f0 + tid + 4 * kThreads * g + kThreads * u, u < 4
  auto note_group = [&](int g, float gx) {
    if constexpr (K > 1) {
      float* p = &s_gm[(g & (kGroupSlots - 1)) * kThreads + tid];
      *p = g < kGroupSlots ? gx : fmaxf(*p, gx);
    }
  };
  if (vec) {
    int64_t f = f0 + tid;
    int g = 0;
    for (; f + 3 * kThreads < f1; f += 4 * kThreads, ++g) {  // four 16-byte loads in flight
      const float4 a = x4[f], b = x4[f + kThreads];
      const float4 c = x4[f + 2 * kThreads], d = x4[f + 3 * kThreads];
      {  // the 16 entries' maximum, one rescale of l, 16 terms: one basic block
        const float4 e[4] = {a, b, c, d};
        float mg = m;
        if constexpr (K > 1) {  // the group's own maximum is kept for the second pass
          float gx = fmaxf(fmaxf(e[0].x, e[0].y), fmaxf(e[0].z, e[0].w));
#pragma unroll
          for (int u = 1; u < 4; ++u) gx = fmaxf(gx, fmaxf(fmaxf(e[u].x, e[u].y), fmaxf(e[u].z, e[u].w)));
          note_group(g, gx);
          mg = fmaxf(m, gx);
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u) mg = fmaxf(mg, fmaxf(fmaxf(e[u].x, e[u].y), fmaxf(e[u].z, e[u].w)));
        }
        float s = l * ptx::ex2((m - mg) * kLog2e);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          s += (ptx::ex2((e[u].x - mg) * kLog2e) + ptx::ex2((e[u].y - mg) * kLog2e)) +
               (ptx::ex2((e[u].z - mg) * kLog2e) + ptx::ex2((e[u].w - mg) * kLog2e));
        l = s;
        m = mg;
      }
      if constexpr (K == 1) {
        const float4 e[4] = {a, b, c, d};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = static_cast<int>(4 * (f + u * kThreads));
          best(e[u].x, j);
          best(e[u].y, j + 1);
          best(e[u].z, j + 2);
          best(e[u].w, j + 3);
        }
      }
    }
    float gt = kNegInf;  // the last (partial, possibly empty) group
    for (; f < f1; f += kThreads) {
      const float4 a = x4[f];
      add4(a);
      gt = fmaxf(gt, fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)));
      const int j = static_cast<int>(4 * f);
      best(a.x, j);
      best(a.y, j + 1);
      best(a.z, j + 2);
      best(a.w, j + 3);
    }
    note_group(g, gt);
  } else {
    for (int64_t j = c0 + tid; j < c1; j += kThreads) {
      const float a = xr[j];
      add1(a);
      best(a, static_cast<int>(j));
    }
  }
  // the running max is the thread's maximum; -inf when it saw only -inf
  // (m never moved and nothing was summed)
  const float tmax = (m > -kMaxFloat || l > 0.f) ? m : kNegInf;

  // warp (m, l)
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off);
    const float lo = __shfl_xor_sync(0xffffffffu, l, off);
    const float mn = fmaxf(m, mo);
    l = l * rebase(m, mn) + lo * rebase(mo, mn);
    m = mn;
  }
  if (lane == 0) {
    s_m[warp] = m;
    s_l[warp] = l;
  }

  List<K> L;
  L.clear();
  float v0;
  int i0;
  if constexpr (K == 1) {
    // the best entry is the thread's argmax; no threshold, no second pass
    __syncthreads();
    if (tid == 0) {  // the CTA's (m, l), read by CTA 0 at the end
      float M = s_m[0], Ls = s_l[0];
      for (int w = 1; w < kWarps; ++w) {
        const float mn = fmaxf(M, s_m[w]);
        Ls = Ls * rebase(M, mn) + s_l[w] * rebase(s_m[w], mn);
        M = mn;
      }
      c_ml[0] = M;
      c_ml[1] = Ls;
    }
    L.v[0] = bv;
    L.i[0] = bi;
  } else {
  // ---- threshold: the K-th largest thread maximum of the warp.  At least K
  // entries of the warp reach it, so an entry below it has K better ones in
  // its own warp and cannot be among the row's K best.
  const float wsorted = warp_sort_desc(tmax);
  float thr = __shfl_sync(0xffffffffu, wsorted, K - 1);  // K <= 32
  if constexpr (K > 16) {
    // a warp's K-th lane maximum is weak for large K: also take the CTA's
    // K-th thread maximum (merged by warp 0); either bound is valid
    // (merged pairwise in log2(kWarps) rounds)
    s_pv[warp * 32 + lane] = wsorted;
#pragma unroll
    for (int step = 1; step < kWarps; step <<= 1) {
      __syncthreads();
      if ((warp & (2 * step - 1)) == 0) {
        const float acc = warp_merge_desc(s_pv[warp * 32 + lane], s_pv[(warp + step) * 32 + lane]);
        __syncwarp();
        s_pv[warp * 32 + lane] = acc;
      }
    }
    __syncthreads();
    if (warp == 0 && lane == 0) c_ml[0] = s_pv[K - 1];  // staged until the summary is written
    __syncthreads();
    thr = fmaxf(thr, c_ml[0]);
  }
  // no CTA barrier here: each warp's second pass needs only its own filter
  // (the CTA's (m, l) is merged after the lists' first barrier)

  // ---- pass 2: entries that beat the filter enter the warp's running best 32
  // (lane-sorted).  The filter starts at (thr, any index) and tightens to the
  // list's K-th entry in the (value, index) order, so later ties and weaker
  // values drop out.  Each round every lane offers one candidate.
  {
    float kv = thr;
    int ki = kNoIndex;
    // A round's candidates (at most one per lane) enter the list one at a
    // time when they are few: each is broadcast, its place is the first lane
    // whose entry it comes before, and the lanes from there on shift up by one
    // (the last entry drops out).  More than eight (a row with many equal
    // maxima, say) are sorted as a batch and merged into the list instead.
    auto round = [&](float cv, int ci) {
      unsigned cl = __ballot_sync(0xffffffffu, ci != kNoIndex);
      if (__popc(cl) > 8) {  // many at once: sort them and merge the batch
        warp_sort_pairs(cv, ci);
        warp_merge_pairs(v0, i0, cv, ci);
        const float nv = __shfl_sync(0xffffffffu, v0, K - 1);
        const int ni = __shfl_sync(0xffffffffu, i0, K - 1);
        if (ni != kNoIndex && before(nv, ni, kv, ki)) {
          kv = nv;
          ki = ni;
        }
        return;
      }
      while (cl) {
        const int src = __ffs(cl) - 1;
        cl &= cl - 1;
        const float v = __shfl_sync(0xffffffffu, cv, src);
        const int j = __shfl_sync(0xffffffffu, ci, src);
        if (!before(v, j, kv, ki)) continue;  // the filter has tightened past it
        const unsigned at = __ballot_sync(0xffffffffu, before(v, j, v0, i0));
        if (at == 0) continue;  // (not reached: v comes before the K-th entry)
        const int pos = __ffs(at) - 1;
        const float uv = __shfl_up_sync(0xffffffffu, v0, 1);
        const int ui = __shfl_up_sync(0xffffffffu, i0, 1);
        if (lane == pos) {
          v0 = v;
          i0 = j;
        } else if (lane > pos) {
          v0 = uv;
          i0 = ui;
        }
        const float nv = __shfl_sync(0xffffffffu, v0, K - 1);
        const int ni = __shfl_sync(0xffffffffu, i0, K - 1);
        if (ni != kNoIndex && before(nv, ni, kv, ki)) {
          kv = nv;
          ki = ni;
        }
      }
    };
    v0 = kNegInf;
    i0 = kNoIndex;
    // The entries of the group at float4 f (when on) that beat the filter are
    // offered to the list, one per lane per round.
    auto offer = [&](int64_t f, bool on) {
      float4 a[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        a[u] = on && f + u * kThreads < f1 ? __ldcs(x4 + f + u * kThreads)
                                           : make_float4(kNegInf, kNegInf, kNegInf, kNegInf);
      uint32_t msk = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        // past the slice: no entry.  Selects instead of a branch measured
        // 2-5 % faster for k <= 16 and 10 % slower at k = 32.
        const bool in = on && f + u * kThreads < f1;
        if constexpr (K <= 16) {
          const uint32_t b = (a[u].x >= kv ? 1u : 0u) | (a[u].y >= kv ? 2u : 0u) |
                             (a[u].z >= kv ? 4u : 0u) | (a[u].w >= kv ? 8u : 0u);
          msk |= (in ? b : 0u) << (4 * u);
        } else {
          if (!in) continue;
          msk |= (a[u].x >= kv ? 1u : 0u) << (4 * u);
          msk |= (a[u].y >= kv ? 2u : 0u) << (4 * u);
          msk |= (a[u].z >= kv ? 4u : 0u) << (4 * u);
          msk |= (a[u].w >= kv ? 8u : 0u) << (4 * u);
        }
      }
      while (__any_sync(0xffffffffu, msk != 0)) {
        float cv = kNegInf;
        int ci = kNoIndex;
        while (msk) {  // this lane's next entry that still beats the filter
          const int e = __ffs(msk) - 1;
          msk &= msk - 1;
          const int u = e >> 2, c = e & 3;
          float4 w = a[0];
          if (u == 1) w = a[1];
          if (u == 2) w = a[2];
          if (u == 3) w = a[3];
          float v = w.x;
          if (c == 1) v = w.y;
          if (c == 2) v = w.z;
          if (c == 3) v = w.w;
          const int j = static_cast<int>(4 * (f + u * kThreads)) + c;
          if (before(v, j, kv, ki)) {
            cv = v;
            ci = j;
            break;
          }
        }
        round(cv, ci);
      }
    };
    if (vec) {
      // Only groups whose maximum reaches thr can hold a candidate.  The warp
      // lists its (lane, slot) pairs that do and shares them out, one per lane
      // per batch of 32, so a warp re-reads a few groups instead of its slice.
      const int ng = static_cast<int>((f1 - f0 + 4 * kThreads - 1) / (4 * kThreads));
      const int nslots = ng < kGroupSlots ? ng : kGroupSlots;
      unsigned my_pm = 0;  // lane s: the lanes whose slot-s groups reach thr
      for (int s = 0; s < nslots; ++s) {
        const unsigned pm = __ballot_sync(0xffffffffu, s_gm[s * kThreads + tid] >= thr);
        if (lane == s) my_pm = pm;
      }
      int incl = __popc(my_pm);  // pairs in slots 0..lane
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      const int trips = (ng + kGroupSlots - 1) / kGroupSlots;  // groups per slot, at most
      for (int t0 = 0; t0 < total; t0 += 32) {
        const int t = t0 + lane;  // this lane's pair
        int slot = 0, skip = 0;   // its slot, and the pairs in the slots before it
        for (int s2 = 0; s2 < nslots; ++s2) {
          const int is = __shfl_sync(0xffffffffu, incl, s2);
          if (is <= t) {
            slot = s2 + 1;
            skip = is;
          }
        }
        const bool task = t < total;
        const unsigned pm = __shfl_sync(0xffffffffu, my_pm, slot & 31);
        const int src = task ? nth_set_bit(pm, t - skip) : 0;
        const int64_t fb = f0 + warp * 32 + src;
        for (int r = 0; r < trips; ++r) {
          const int gg = slot + r * kGroupSlots;
          offer(fb + static_cast<int64_t>(4 * kThreads) * gg, task && gg < ng);
        }
      }
    } else {
      for (int64_t j0 = c0; j0 < c1; j0 += kThreads) {
        const int64_t j = j0 + tid;
        const float a = j < c1 ? __ldcs(xr + j) : kNegInf;
        const bool cand = j < c1 && before(a, static_cast<int>(j), kv, ki);
        if (__any_sync(0xffffffffu, cand))
          round(cand ? a : kNegInf, cand ? static_cast<int>(j) : kNoIndex);
      }
    }
  }
  }  // K > 1
  if constexpr (K == 1) {
    cluster_topk<K>(L, s_pv, s_pi, c_v, c_i, nct, rank, v0, i0);
  } else {
    cluster_merge_lists(v0, i0, s_pv, s_pi, s_m, s_l, c_ml, c_v, c_i, nct, rank);
  }
  if (rank == 0 && warp == 0) {
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
  }
  if (nct > 1) cluster_sync_all();  // CTA 0 has read every CTA's shared memory
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
