// attn_bwd.cu — exact softmax attention backward on sm_103a tensor cores.
//
// "Online softmax" (zerotofrontier.app), "From weights to outputs": the
// log-sum-exp kept by the forward pass is all the backward pass needs to
// rebuild the weights, y_j = exp(s_j - lse).  With s = scale * q.k,
// P = exp(s - lse) (0 where masked), dO the gradient of the output O:
//   dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,
//   dS = P * (dP - D)  (elementwise, D broadcast along each row),
//   dQ = scale * dS K,  dK = scale * dS^T Q.
// The score and weight matrices are rebuilt tile by tile and never stored.
//
// Three kernels:
//   bwd_delta_kernel  D = rowsum(dO * O), fp32 (HBM-bound).
//   bwd_dq_kernel     one CTA per (b, h, 128-query tile); streams the visible
//                     K tiles (three slots) and V tiles (one slot).  S = Q K^T
//                     and dP = dO V^T into TMEM; two threads per query row
//                     (each half the columns) form P and dS (lse and D in
//                     registers) and write dS as bf16 over the S columns;
//                     dQ += dS K with dS read straight from TMEM.
//   bwd_dkdv_kernel   one CTA per (b, h, 128-key tile); streams (Q_i, dO_i)
//                     pairs for the query tiles that see it.  S^T = K Q^T and
//                     dP^T = V dO^T into TMEM; two threads per key row form
//                     P^T and dS^T (lse and D per column from shared memory)
//                     and write both as bf16 over S^T and dP^T; dV += P^T dO
//                     and dK += dS^T Q read them straight from TMEM.
// dQ and dK/dV are separate so that no partial sum crosses CTAs (no atomics);
// the price is S and dP formed twice (7 instead of 5 matrix products).  The
// outputs leave through bulk tensor stores of boxes that each warp stages in
// the ring's shared memory, idle once the last product has completed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace osm {
namespace bwd {

using namespace ptx;

constexpr int kTile = 128;   // rows of every tile (query or key)
constexpr int kSlots = 4;    // streamed 32 KB tiles in flight
constexpr int kPairs = kSlots / 2;  // dK/dV kernel: the slots as (Q_i, dO_i) pairs
constexpr uint32_t kKSlots = 3, kVSlot = 3;  // dQ kernel: K tiles in slots 0-2, V in slot 3
constexpr uint32_t kTileBytes = kTile * 128 * 2;  // 32768: a slot holds a d = 128 tile
constexpr uint32_t kBoxBytes = 128 * 64 * 2;           // one TMA box: 64 columns x 128 rows
constexpr int kThreads = 384;  // warp 0 TMA, warp 1 MMA, warps 4-11 element-wise
// The element-wise warps: two per TMEM lane quarter, warp 4 + q + 4h takes
// columns 64h .. 64h+63 of rows 32q .. 32q+31.  Each writes its packed bf16
// results inside its own half (chunk c of 32 columns at 64(c/2) + 16(c%2)),
// so neither overwrites columns the other has not read yet; the products that
// read them address 16-column step kk at tmem_half_col(kk).
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kPosInf = __builtin_huge_valf();

// shared memory: two resident tiles, then the ring
constexpr uint32_t kSmemRes = 0;
constexpr uint32_t kSmemRing = 2 * kTileBytes;
constexpr uint32_t kSmemBar = kSmemRing + kSlots * kTileBytes;
enum Bar : uint32_t {
  RES_FULL = 0,
  RING_FULL = 1,                 // [kSlots]
  RING_EMPTY = 1 + kSlots,       // [kSlots]
  S_FULL = 1 + 2 * kSlots,
  P_FULL = S_FULL + 1,
  O_FULL = P_FULL + 1,
  DRAIN = O_FULL + 1,
  DP_FULL = DRAIN + 1,   // dK/dV kernel: dP^T ready (S_FULL then only S^T)
  DS_FULL = DP_FULL + 1, // dS (dS^T) written
  S_FULL1 = DS_FULL + 1, // dQ kernel: the second S buffer ready
  NUM_BARS
};
constexpr uint32_t kSmemTmemSlot = kSmemBar + 8 * NUM_BARS;
constexpr uint32_t kSmemAbort = kSmemTmemSlot + 4;
// per softmax warp: [2 buffers][lse2 | D][128 columns] floats
constexpr uint32_t kSmemCol = (kSmemAbort + 4 + 15) / 16 * 16;
constexpr uint32_t kColFloats = 2 * 2 * (kTile / 2);
// The outputs leave through the ring, idle once every product has completed:
// each element-wise warp stages its 32 rows there (at most 8 KB) for bulk
// tensor stores.
constexpr uint32_t kSmemBytes = kSmemCol + 8 * kColFloats * 4 + 1024;  // + alignment slack

constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemAcc0 = 256, kTmemAcc1 = 384;

constexpr uint32_t kIdescKK = idesc_bf16_f32(128, 128, false);  // both operands K-major

constexpr unsigned kSiteQ = 0x02000000u;   // error-word sites of the dQ kernel
constexpr unsigned kSiteK = 0x03000000u;   // ... and of the dK/dV kernel
constexpr unsigned kChk = 0x0E040000u;     // index checks of an OSM_CHECKED build

struct Params {
  int B, H, Nq, Nk;
  int causal;
  int n_qt, n_kt;     // query / key tiles per head
  float scale, scale_log2;
  const int32_t* key_len;
  const float* lse;   // [B*H*Nq] natural log
  const float* delta; // [B*H*Nq]
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  unsigned int* err;
};

__device__ __forceinline__ int key_len_of(const Params& p, int b) {
  int L = p.key_len ? p.key_len[b] : p.Nk;
  return L < 0 ? 0 : (L > p.Nk ? p.Nk : L);
}

__host__ __device__ constexpr uint32_t tmem_half_col(int kk) {
  return static_cast<uint32_t>(64 * (kk >> 2) + 8 * (kk & 3));
}

// A warp's 32 accumulator rows (this thread's row in r, N fp32 columns, times
// mul) as bf16 in a shared-memory stage laid out for bulk tensor stores:
// N / 64 boxes of 32 rows x 64 columns (4 KB each), 128 bytes a row, the
// 16-byte pieces in the 128-byte swizzle (piece e of row r at e ^ (r & 7)),
// so the lanes' writes meet no bank twice.  The stage is 1024-byte aligned.
template <int N>
__device__ __forceinline__ void stage_rows_sw128(const uint32_t (&r)[N], float mul, uint8_t* stage) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int h = 0; h < N / 64; ++h) {
    uint4* srow = reinterpret_cast<uint4*>(stage + 4096 * h + 128 * lane);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      uint32_t w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(r[64 * h + 8 * e + 2 * u]) * mul,
                                                  __uint_as_float(r[64 * h + 8 * e + 2 * u + 1]) * mul);
        w[u] = *reinterpret_cast<uint32_t*>(&h2);
      }
      srow[e ^ (lane & 7)] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}
// The same for 32 columns: one box of 32 rows x 32 columns, 64 bytes a row,
// no swizzle.
__device__ __forceinline__ void stage_rows_32(const uint32_t (&r)[32], float mul, uint8_t* stage) {
  const int lane = threadIdx.x & 31;
  uint4* srow = reinterpret_cast<uint4*>(stage + 64 * lane);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    uint32_t w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(r[8 * e + 2 * u]) * mul,
                                                __uint_as_float(r[8 * e + 2 * u + 1]) * mul);
      w[u] = *reinterpret_cast<uint32_t*>(&h2);
    }
    srow[e] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <int D>
__device__ __forceinline__ void zero_row_bf16(__nv_bfloat16* dst) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int e = 0; e < D / 8; ++e) d4[e] = make_uint4(0, 0, 0, 0);
}

__device__ unsigned int g_bwd_err;

// ------------------------------------------------------------------ D
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                        const __nv_bfloat16* __restrict__ dout,
                                                        float* __restrict__ delta, int64_t rows) {
  // D/8 lanes per row, 8 columns (one 16-byte load of each tensor) per lane
  constexpr int kLanes = D / 8;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = t / kLanes;
  const int sl = threadIdx.x % kLanes;
  float acc = 0.f;
  if (row < rows) {
    const uint4 a = reinterpret_cast<const uint4*>(o + row * D)[sl];
    const uint4 g = reinterpret_cast<const uint4*>(dout + row * D)[sl];
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wg[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(wa[i] << 16), __uint_as_float(wg[i] << 16), acc);
      acc = fmaf(__uint_as_float(wa[i] & 0xffff0000u), __uint_as_float(wg[i] & 0xffff0000u), acc);
    }
  }
#pragma unroll
  for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && sl == 0) delta[row] = acc;
}

// ------------------------------------------------------------------ dQ
// Item = (bh, query tile); causal items longest first.  D: head dimension.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array, so that
  // accesses through it compile to shared-memory instructions (an integer
  // round trip of the address leaves them generic, which measured 8 % slower)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + kSmemRes, sDO = sQ + kTileBytes, sRing = sbase + kSmemRing;
  auto bar = [&](uint32_t i) { return sbase + kSmemBar + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemTmemSlot);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int within = blockIdx.x % p.n_qt;
  const int bh = blockIdx.x / p.n_qt;
  const int qt = p.causal ? (p.n_qt - 1 - within) : within;
  const int q0 = qt * kTile;
  const int b = bh / p.H;
  const int L = key_len_of(p, b);
  int kend = L;
  if (p.causal) kend = min(L, max(0, min(q0 + kTile, p.Nq) + (p.Nk - p.Nq)));
  const int n_kv = (kend + kTile - 1) / kTile;

  if (n_kv == 0) {  // no visible key for any row of the tile: dQ = 0
    if (warp >= 4 && warp < 8) {
      const int row = q0 + 32 * (warp - 4) + lane;
      if (row < p.Nq && checked(bh < p.B * p.H, p.err, kChk | 1))
        zero_row_bf16<D>(p.dq + (static_cast<int64_t>(bh) * p.Nq + row) * D);
    }
    return;
  }

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(RES_FULL), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(RING_FULL + s), 1);
      mbar_init(bar(RING_EMPTY + s), 1);
    }
    mbar_init(bar(S_FULL), 1);
    mbar_init(bar(S_FULL1), 1);
    mbar_init(bar(DP_FULL), 1);
    mbar_init(bar(DS_FULL), 8);
    mbar_init(bar(O_FULL), 1);
    mbar_init(bar(DRAIN), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  auto wait_one = [&](uint32_t bb, uint32_t parity, unsigned site) -> bool {
    return wait_bounded(bb, parity, abort_flag, p.err, site);
  };

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------- TMA producer
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_do);
    mbar_arrive_expect_tx(bar(RES_FULL), 2 * kTile * D * 2);
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(sQ + c * kBoxBytes, &tm_q, bar(RES_FULL), c * 64, q0, bh);
      tma_load_3d(sDO + c * kBoxBytes, &tm_do, bar(RES_FULL), c * 64, q0, bh);
    }
    // K tiles through slots 0-2 and V tiles through slot 3, loaded in the
    // order K_0, V_0, K_1, then (K_{j+2}, V_{j+1}) for j = 0, 1, ...: K_j is
    // read by S_j (issued in step j-1) and by dQ_j (step j), V_j only by dP_j,
    // so three K slots let K_{j+2} load while step j-1 runs.
    uint32_t kslot = 0, kph = 0, vph = 0, fill_mask = 0, fill_ph = 0;
    bool ok = true;
    auto load = [&](uint32_t sl, uint32_t phs, const CUtensorMap* tm, int j) -> bool {
      if (!wait_one(bar(RING_EMPTY + sl), phs ^ 1, kSiteQ | 1)) return false;
      mbar_arrive_expect_tx(bar(RING_FULL + sl), kTile * D * 2);
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(sRing + sl * kTileBytes + c * kBoxBytes, tm, bar(RING_FULL + sl), c * 64,
                    j * kTile, bh);
      fill_mask |= 1u << sl;
      fill_ph = (fill_ph & ~(1u << sl)) | (phs << sl);
      return true;
    };
    auto load_k = [&](int j) -> bool {
      const bool r = load(kslot, kph, &tm_k, j);
      if (++kslot == kKSlots) { kslot = 0; kph ^= 1; }
      return r;
    };
    auto load_v = [&](int j) -> bool {
      const bool r = load(kVSlot, vph, &tm_v, j);
      vph ^= 1;
      return r;
    };
    if (n_kv > 0) ok = load_k(0) && load_v(0);
    if (ok && n_kv > 1) ok = load_k(1);
    for (int j = 0; ok && j + 1 < n_kv; ++j) {
      if (j + 2 < n_kv) ok = load_k(j + 2);
      if (ok) ok = load_v(j + 1);
    }
    if (!ok) {  // let every copy this thread started land before the CTA exits
      for (int s = 0; s < kSlots; ++s)
        if (fill_mask >> s & 1u) wait_drain(bar(RING_FULL + s), fill_ph >> s & 1u, 200000000ull);
      wait_drain(bar(RES_FULL), 0, 200000000ull);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs this loop (its descriptor arithmetic stays
    // warp-uniform); one elected lane issues each MMA and commit.
    auto wait_w = [&](uint32_t bb, uint32_t parity, unsigned site) -> bool {
      return __all_sync(0xffffffffu, wait_one(bb, parity, site));
    };
    auto commit = [&](uint32_t bb) {
      if (elect_one()) mma_commit(bb);
      __syncwarp();
    };
    // S is double-buffered (TMEM columns 0 and 384): order per key tile j is
    // S_{j+1} | dQ += dS_j K_j (after dS_j) | dP_{j+1}, so S_{j+1} runs while
    // the element-wise warps work on tile j.  Every product that overwrites a
    // TMEM region is issued after the product that reads it.
    const uint64_t dKm = sdesc_sw128(0, 16, 1024);      // K-major template
    const uint64_t dMN = sdesc_sw128(0, 16384, 1024);   // MN-major template
    bool ok = wait_w(bar(RES_FULL), 0, kSiteQ | 2);
    uint32_t kslot = 0, kph = 0, vph = 0, df_ph = 0;
    if (ok) {
      tc_fence_after();
      const uint64_t qdesc = dKm + (sQ >> 4), dodesc = dKm + (sDO >> 4);
      auto next_k = [&](uint32_t& s_out) -> bool {  // K slots in fill order
        s_out = kslot;
        const bool r = wait_w(bar(RING_FULL + kslot), kph, kSiteQ | 4);
        if (++kslot == kKSlots) { kslot = 0; kph ^= 1; }
        return r;
      };
      auto next_v = [&](uint32_t& s_out) -> bool {
        s_out = kVSlot;
        const bool r = wait_w(bar(RING_FULL + kVSlot), vph, kSiteQ | 4);
        vph ^= 1;
        return r;
      };
      auto issue_s = [&](uint32_t ks, int jj) {  // S_jj = Q K_jj^T into buffer jj & 1
        tc_fence_after();
        const uint64_t kdesc = dKm + ((sRing + ks * kTileBytes) >> 4);
        const uint32_t tsb = tbase + ((jj & 1) ? kTmemAcc1 : kTmemS);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
          if (elect_one()) mma_ss(tsb, qdesc + off, kdesc + off, kIdescKK, kk > 0 ? 1u : 0u);
          __syncwarp();
        }
        commit(bar((jj & 1) ? S_FULL1 : S_FULL));
      };
      auto issue_dp = [&](uint32_t vs) {  // dP = dO V_j^T; V_j is used by dP_j only
        tc_fence_after();
        const uint64_t vdesc = dKm + ((sRing + vs * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
          if (elect_one()) mma_ss(tbase + kTmemDP, dodesc + off, vdesc + off, kIdescKK, kk > 0 ? 1u : 0u);
          __syncwarp();
        }
        commit(bar(DP_FULL));
        commit(bar(RING_EMPTY + vs));
      };
      uint32_t ks = 0, vs = 0;
      if ((ok = next_k(ks))) issue_s(ks, 0);
      if (ok && (ok = next_v(vs))) issue_dp(vs);
      for (int j = 0; ok && j < n_kv; ++j) {
        const bool more = j + 1 < n_kv;
        uint32_t kn = 0;
        if (more) {
          if (!(ok = next_k(kn))) break;
          issue_s(kn, j + 1);
        }
        // dQ += dS_j K_j once the element-wise warps have written dS_j
        if (!(ok = wait_w(bar(DS_FULL), df_ph, kSiteQ | 3))) break;
        df_ph ^= 1;
        tc_fence_after();
        const uint64_t kdesc = dMN + ((sRing + ks * kTileBytes) >> 4);
        const uint32_t tsb = tbase + ((j & 1) ? kTmemAcc1 : kTmemS);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          if (elect_one())
            mma_ts(tbase + kTmemAcc0, tsb + tmem_half_col(kk), kdesc + ((kk * 2048) >> 4),
                   idesc_bf16_f32(128, D, true), (j > 0 || kk > 0) ? 1u : 0u);
          __syncwarp();
        }
        commit(bar(RING_EMPTY + ks));  // K_j is free after this product
        if (more) {
          if (!(ok = next_v(vs))) break;
          issue_dp(vs);
        }
        ks = kn;
      }
      if (ok) commit(bar(O_FULL));
    }
    if (!ok) {  // wait for every MMA already issued before TMEM is released
      commit(bar(DRAIN));
      if (lane == 0) wait_drain(bar(DRAIN), 0, 200000000ull);
      __syncwarp();
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------- P and dS
    const int wq = warp & 3, hh = (warp - 4) >> 2;  // lane quarter, column half
    const uint32_t lane_off = static_cast<uint32_t>(32 * wq) << 16;
    const uint32_t tDP = tbase + lane_off + kTmemDP;
    const int row = q0 + 32 * wq + lane;
    const bool row_ok = row < p.Nq;
    const int64_t grow = static_cast<int64_t>(bh) * p.Nq + (row_ok ? row : 0);
    float lse2 = row_ok ? p.lse[grow] * kLog2e : kPosInf;
    if (!(lse2 > kNegInf)) lse2 = kPosInf;  // a row with no visible key: every P is 0
    const float dlt = row_ok ? p.delta[grow] : 0.f;
    const float nlse2 = -lse2, ndlt = -dlt;
    int limit = L;
    if (p.causal) limit = min(limit, row + 1 + (p.Nk - p.Nq));
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      // phase A: P from S_j (buffer j & 1), kept in fp32 registers
      const uint32_t tSb = tbase + lane_off + ((j & 1) ? kTmemAcc1 : kTmemS);
      ok = __all_sync(0xffffffffu,
                      wait_one(bar((j & 1) ? S_FULL1 : S_FULL), (j >> 1) & 1, kSiteQ | 5));
      if (!ok) break;
      tc_fence_after();
      const int k0 = j * kTile;
      const bool masked_tile = __any_sync(0xffffffffu, k0 + kTile > limit);
      float pr[2][32];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int ch = 2 * hh + c;
        uint32_t sv[32];
        tmem_ld_x32(tSb + 32 * ch, sv);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float x0, x1;
          fma2(x0, x1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), sl2, sl2, nlse2, nlse2);
          pr[c][e] = ex2(x0);
          pr[c][e + 1] = ex2(x1);
        }
        if (masked_tile) {  // after the chunk, so the loop above stays one basic block
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (k0 + 32 * ch + e >= limit) pr[c][e] = 0.f;
        }
      }
      // phase B: dS = P (dP - D), written as bf16 over this half of S_j
      ok = __all_sync(0xffffffffu, wait_one(bar(DP_FULL), j & 1, kSiteQ | 7));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int ch = 2 * hh + c;
        uint32_t dp[32], pk[16];
        tmem_ld_x32(tDP + 32 * ch, dp);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float t0 = __uint_as_float(dp[e]), t1 = __uint_as_float(dp[e + 1]), g0, g1;
          add2(t0, t1, ndlt, ndlt);  // dP - D
          fma2(g0, g1, t0, t1, pr[c][e], pr[c][e + 1], 0.f, 0.f);
          __nv_bfloat162 h2 = __floats2bfloat162_rn(g0, g1);
          pk[e >> 1] = *reinterpret_cast<uint32_t*>(&h2);
        }
        tmem_st_x16_nowait(tSb + 64 * hh + 16 * c, pk);  // over this half's S_j, already read
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(DS_FULL));
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_one(bar(O_FULL), 0, kSiteQ | 6));
    if (ok) {
      tc_fence_after();
      const int row0 = row - lane;  // the warp's first query row
      // this warp's half of its rows' dQ (D / 2 columns) staged in the idle
      // ring and stored as one box; rows past Nq are not written, and a warp
      // whose rows all lie past Nq stores nothing
      constexpr int kHalf = D / 2;
      uint8_t* stage = smem + kSmemRing + (warp - 4) * (32 * kHalf * 2);
      uint32_t r[kHalf];
      tmem_ld_cols<kHalf>(tbase + lane_off + kTmemAcc0 + hh * kHalf, r);
      if constexpr (kHalf == 64) stage_rows_sw128<kHalf>(r, p.scale, stage);
      else stage_rows_32(r, p.scale, stage);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && row0 < p.Nq && checked(bh < p.B * p.H && row0 >= 0, p.err, kChk | 2)) {
        tma_store_3d(&tm_dq, smem_u32(stage), hh * kHalf, row0, bh);
        bulk_wait_read_0();  // the box has left shared memory before the CTA ends
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// ------------------------------------------------------------------ dK, dV
// Item = (bh, key tile); causal items longest first (early key tiles are
// seen by the most query tiles).  D: head dimension.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_dk,
                    const __grid_constant__ CUtensorMap tm_dv, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned by pointer arithmetic on the shared array, so that
  // accesses through it compile to shared-memory instructions (an integer
  // round trip of the address leaves them generic, which measured 8 % slower)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase + kSmemRes, sV = sK + kTileBytes, sRing = sbase + kSmemRing;
  auto bar = [&](uint32_t i) { return sbase + kSmemBar + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemTmemSlot);
  float* col = reinterpret_cast<float*>(smem + kSmemCol);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int kt = blockIdx.x % p.n_kt;  // causal: key tile 0 first (it has the most work)
  const int bh = blockIdx.x / p.n_kt;
  const int k0 = kt * kTile;
  const int b = bh / p.H;
  const int L = key_len_of(p, b);
  const int off = p.Nk - p.Nq;
  int qt_first = 0;
  if (p.causal) qt_first = max(0, k0 - off) / kTile;
  const int n_q = (k0 < L && (!p.causal || k0 - off < p.Nq)) ? p.n_qt - qt_first : 0;

  if (n_q == 0) {  // every key of the tile is invisible to every query: dK = dV = 0
    if (warp >= 4 && warp < 8) {
      const int key = k0 + 32 * (warp - 4) + lane;
      if (key < p.Nk && checked(bh < p.B * p.H, p.err, kChk | 3)) {
        const int64_t g = (static_cast<int64_t>(bh) * p.Nk + key) * D;
        zero_row_bf16<D>(p.dk + g);
        zero_row_bf16<D>(p.dv + g);
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(RES_FULL), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(RING_FULL + s), 1);
      mbar_init(bar(RING_EMPTY + s), 1);
    }
    mbar_init(bar(S_FULL), 1);
    mbar_init(bar(DP_FULL), 1);
    mbar_init(bar(P_FULL), 8);
    mbar_init(bar(DS_FULL), 8);
    mbar_init(bar(O_FULL), 1);
    mbar_init(bar(DRAIN), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  auto wait_one = [&](uint32_t bb, uint32_t parity, unsigned site) -> bool {
    return wait_bounded(bb, parity, abort_flag, p.err, site);
  };

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------- TMA producer
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_do);
    mbar_arrive_expect_tx(bar(RES_FULL), 2 * kTile * D * 2);
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(sK + c * kBoxBytes, &tm_k, bar(RES_FULL), c * 64, k0, bh);
      tma_load_3d(sV + c * kBoxBytes, &tm_v, bar(RES_FULL), c * 64, k0, bh);
    }
    // (Q_i, dO_i) as one pair of slots under one barrier: both are read by
    // query tile i's products and released together after dK_i
    uint32_t slot = 0, ph = 0, fill_mask = 0, fill_ph = 0;
    bool ok = true;
    for (int i = 0; ok && i < n_q; ++i) {
      const int qrow = (qt_first + i) * kTile;
      if (!(ok = wait_one(bar(RING_EMPTY + slot), ph ^ 1, kSiteK | 1))) break;
      mbar_arrive_expect_tx(bar(RING_FULL + slot), 2 * kTile * D * 2);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(sRing + (2 * slot) * kTileBytes + c * kBoxBytes, &tm_q, bar(RING_FULL + slot),
                    c * 64, qrow, bh);
        tma_load_3d(sRing + (2 * slot + 1) * kTileBytes + c * kBoxBytes, &tm_do,
                    bar(RING_FULL + slot), c * 64, qrow, bh);
      }
      fill_mask |= 1u << slot;
      fill_ph = (fill_ph & ~(1u << slot)) | (ph << slot);
      if (++slot == kPairs) { slot = 0; ph ^= 1; }
    }
    if (!ok) {
      for (int s = 0; s < kPairs; ++s)
        if (fill_mask >> s & 1u) wait_drain(bar(RING_FULL + s), fill_ph >> s & 1u, 200000000ull);
      wait_drain(bar(RES_FULL), 0, 200000000ull);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs this loop (its descriptor arithmetic stays
    // warp-uniform); one elected lane issues each MMA and commit.
    auto wait_w = [&](uint32_t bb, uint32_t parity, unsigned site) -> bool {
      return __all_sync(0xffffffffu, wait_one(bb, parity, site));
    };
    auto commit = [&](uint32_t bb) {
      if (elect_one()) mma_commit(bb);
      __syncwarp();
    };
    // Order per query tile i: S_i, dP_i | dV_i (after P_i) | S_{i+1} | dK_i
    // (after dS_i) | dP_{i+1}.  Each element-wise phase overlaps two products,
    // and every product that overwrites a TMEM region is issued after the
    // product that reads it (the tensor pipe runs them in issue order).
    const uint64_t dKm = sdesc_sw128(0, 16, 1024);
    const uint64_t dMN = sdesc_sw128(0, 16384, 1024);
    bool ok = wait_w(bar(RES_FULL), 0, kSiteK | 2);
    uint32_t slot = 0, ph = 0, pf_ph = 0, df_ph = 0;
    if (ok) {
      tc_fence_after();
      const uint64_t kdesc = dKm + (sK >> 4), vdesc = dKm + (sV >> 4);
      // pair p holds Q_i in slot 2p and dO_i in slot 2p + 1
      auto next_pair = [&](uint32_t& p_out) -> bool {
        p_out = slot;
        const bool r = wait_w(bar(RING_FULL + slot), ph, kSiteK | 4);
        if (++slot == kPairs) { slot = 0; ph ^= 1; }
        return r;
      };
      auto issue_s = [&](uint32_t qs) {  // S^T = K Q_i^T
        tc_fence_after();
        const uint64_t qdesc = dKm + ((sRing + qs * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o16 = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
          if (elect_one()) mma_ss(tbase + kTmemS, kdesc + o16, qdesc + o16, kIdescKK, kk > 0 ? 1u : 0u);
          __syncwarp();
        }
        commit(bar(S_FULL));
      };
      auto issue_dp = [&](uint32_t ds) {  // dP^T = V dO_i^T
        tc_fence_after();
        const uint64_t dodesc = dKm + ((sRing + ds * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o16 = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
          if (elect_one()) mma_ss(tbase + kTmemDP, vdesc + o16, dodesc + o16, kIdescKK, kk > 0 ? 1u : 0u);
          __syncwarp();
        }
        commit(bar(DP_FULL));
      };
      uint32_t pc = 0;
      if ((ok = next_pair(pc))) {
        issue_s(2 * pc);
        issue_dp(2 * pc + 1);
      }
      for (int i = 0; ok && i < n_q; ++i) {
        const bool more = i + 1 < n_q;
        const uint32_t qs = 2 * pc, ds = 2 * pc + 1;
        uint32_t pn = 0;
        // dV += P_i^T dO_i once the element-wise warps have written P_i
        if (!(ok = wait_w(bar(P_FULL), pf_ph, kSiteK | 3))) break;
        pf_ph ^= 1;
        tc_fence_after();
        const uint64_t dod = dMN + ((sRing + ds * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          if (elect_one())
            mma_ts(tbase + kTmemAcc0, tbase + kTmemS + tmem_half_col(kk), dod + ((kk * 2048) >> 4),
                   idesc_bf16_f32(128, D, true), (i > 0 || kk > 0) ? 1u : 0u);
          __syncwarp();
        }
        if (more) {
          if (!(ok = next_pair(pn))) break;
          issue_s(2 * pn);
        }
        // dK += dS_i^T Q_i once they have written dS_i
        if (!(ok = wait_w(bar(DS_FULL), df_ph, kSiteK | 7))) break;
        df_ph ^= 1;
        tc_fence_after();
        const uint64_t qd = dMN + ((sRing + qs * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          if (elect_one())
            mma_ts(tbase + kTmemAcc1, tbase + kTmemDP + tmem_half_col(kk), qd + ((kk * 2048) >> 4),
                   idesc_bf16_f32(128, D, true), (i > 0 || kk > 0) ? 1u : 0u);
          __syncwarp();
        }
        commit(bar(RING_EMPTY + pc));  // Q_i and dO_i are free after dK_i
        if (more) issue_dp(2 * pn + 1);
        pc = pn;
      }
      if (ok) commit(bar(O_FULL));
    }
    if (!ok) {
      commit(bar(DRAIN));
      if (lane == 0) wait_drain(bar(DRAIN), 0, 200000000ull);
      __syncwarp();
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------- P^T and dS^T
    const int wq = warp & 3, hh = (warp - 4) >> 2;  // lane quarter, column half
    const int tid = 32 * wq + lane;  // 0..127: this thread's key row
    const uint32_t lane_off = static_cast<uint32_t>(32 * wq) << 16;
    const uint32_t tS = tbase + lane_off + kTmemS, tDP = tbase + lane_off + kTmemDP;
    const int key = k0 + tid;
    const bool key_ok = key < L;  // keys past the valid length see no query
    const float sl2 = p.scale_log2;
    const int64_t hrow = static_cast<int64_t>(bh) * p.Nq;
    // Per-column lse (base 2) and D of this warp's 64 columns of query tile i.
    // Every warp stages its own copy in shared memory (lane l loads columns
    // 2l, 2l+1 of its half), so only __syncwarp is needed; the next tile's
    // values load while this one runs.
    float* colw = col + (warp - 4) * kColFloats;
    // The raw lse and D are loaded a tile ahead and converted where they are
    // staged, so the global loads' latency is never waited on.
    auto col_vals = [&](int i, float (&l2)[2], float (&dd)[2]) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int q = (qt_first + i) * kTile + 64 * hh + 2 * lane + u;
        const bool in = q < p.Nq;
        l2[u] = in ? p.lse[hrow + q] : kNegInf;
        dd[u] = in ? p.delta[hrow + q] : 0.f;
      }
    };
    float nl2[2], nd[2];
    col_vals(0, nl2, nd);
    uint32_t sf_ph = 0;
    bool ok = true;
    for (int i = 0; i < n_q; ++i) {
      float* cl = colw + (i & 1) * kTile;  // [lse2 | D] x 64 columns
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        // stored negated: -lse2 and -D enter packed adds directly; a query
        // with no visible key (lse -inf) gets -lse2 = -inf, so P = 0
        const float nl = -nl2[u] * kLog2e;
        cl[2 * lane + u] = nl < kPosInf ? nl : kNegInf;
        cl[kTile / 2 + 2 * lane + u] = -nd[u];
      }
      __syncwarp();
      if (i + 1 < n_q) col_vals(i + 1, nl2, nd);
      // phase A: P^T from S^T, kept in fp32 registers, written as bf16 over S^T
      ok = __all_sync(0xffffffffu, wait_one(bar(S_FULL), sf_ph, kSiteK | 5));
      if (!ok) break;
      sf_ph ^= 1;
      tc_fence_after();
      const int qb = (qt_first + i) * kTile;
      // the tile needs the causal mask when some (key, query) pair is hidden
      const bool masked_tile = p.causal && __any_sync(0xffffffffu, key > qb + off);
      const bool need_mask = masked_tile || __any_sync(0xffffffffu, !key_ok);
      float pr[2][32];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int ch = 2 * hh + c;
        uint32_t sv[32], pk[16];
        tmem_ld_x32(tS + 32 * ch, sv);
        const float4* cl4 = reinterpret_cast<const float4*>(cl + 32 * c);
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 l4 = cl4[e4];  // -lse2 of four columns
          const int e = 4 * e4;
          float x[4];
          fma2(x[0], x[1], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), sl2, sl2, l4.x, l4.y);
          fma2(x[2], x[3], __uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3]), sl2, sl2, l4.z, l4.w);
#pragma unroll
          for (int u = 0; u < 4; ++u) pr[c][e + u] = ex2(x[u]);
        }
        // the mask after the whole chunk: the loop above stays one basic
        // block (a branch per group of four measured twice as slow)
        if (need_mask) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (!key_ok || (masked_tile && key > qb + 32 * ch + e + off)) pr[c][e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          __nv_bfloat162 h2 = __floats2bfloat162_rn(pr[c][2 * e], pr[c][2 * e + 1]);
          pk[e] = *reinterpret_cast<uint32_t*>(&h2);
        }
        tmem_st_x16_nowait(tS + 64 * hh + 16 * c, pk);  // over this half's S^T, already read
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(P_FULL));
      // phase B: dS^T = P^T (dP^T - D), written as bf16 over dP^T
      ok = __all_sync(0xffffffffu, wait_one(bar(DP_FULL), sf_ph ^ 1, kSiteK | 8));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int ch = 2 * hh + c;
        uint32_t dp[32], gk[16];
        tmem_ld_x32(tDP + 32 * ch, dp);
        const float4* cd4 = reinterpret_cast<const float4*>(cl + kTile / 2 + 32 * c);
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 d4 = cd4[e4];  // -D of four columns
          const int e = 4 * e4;
          float t[4], g[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) t[u] = __uint_as_float(dp[e + u]);
          add2(t[0], t[1], d4.x, d4.y);  // dP - D
          add2(t[2], t[3], d4.z, d4.w);
          fma2(g[0], g[1], t[0], t[1], pr[c][e], pr[c][e + 1], 0.f, 0.f);
          fma2(g[2], g[3], t[2], t[3], pr[c][e + 2], pr[c][e + 3], 0.f, 0.f);
          __nv_bfloat162 g0 = __floats2bfloat162_rn(g[0], g[1]);
          __nv_bfloat162 g1 = __floats2bfloat162_rn(g[2], g[3]);
          gk[2 * e4] = *reinterpret_cast<uint32_t*>(&g0);
          gk[2 * e4 + 1] = *reinterpret_cast<uint32_t*>(&g1);
        }
        tmem_st_x16_nowait(tDP + 64 * hh + 16 * c, gk);  // over this half's dP^T, already read
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(DS_FULL));
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_one(bar(O_FULL), 0, kSiteK | 6));
    if (ok) {
      tc_fence_after();
      const int key0 = key - lane;  // the warp's first key row
      // this warp's rows of dV (hh = 0) or dK (hh = 1) staged in the idle
      // ring and stored as D / 64 boxes; rows past Nk are not written
      uint8_t* stage = smem + kSmemRing + (warp - 4) * (32 * D * 2);
      uint32_t r[D];
      tmem_ld_row<D>(tbase + lane_off + (hh == 0 ? kTmemAcc0 : kTmemAcc1), r);
      stage_rows_sw128<D>(r, hh == 0 ? 1.f : p.scale, stage);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && key0 < p.Nk && checked(bh < p.B * p.H && key0 >= 0, p.err, kChk | 4)) {
#pragma unroll
        for (int h = 0; h < D / 64; ++h)
          tma_store_3d(hh == 0 ? &tm_dv : &tm_dk, smem_u32(stage) + 4096 * h, 64 * h, key0, bh);
        bulk_wait_read_0();  // the boxes have left shared memory before the CTA ends
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

}  // namespace bwd

size_t attn_bwd_workspace_bytes(int B, int H, int Nq) {
  return ((static_cast<size_t>(B) * H * Nq * 4 + 255) / 256) * 256;
}

cudaError_t launch_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dout, void* dq, void* dk, void* dv,
                            int B, int H, int Nq, int Nk, int d, float scale, int causal,
                            const int32_t* key_len, void* workspace, cudaStream_t s,
                            bool* tmap_ok) {
  using namespace bwd;
  *tmap_ok = true;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t qrows = BH * Nq;
  float* delta = static_cast<float*>(workspace);
  if (Nq > 0) {
    const unsigned nb = static_cast<unsigned>((qrows * (d / 8) + 255) / 256);
    if (d == 128)
      bwd_delta_kernel<128><<<nb, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(o),
                                               static_cast<const __nv_bfloat16*>(dout), delta,
                                               qrows);
    else
      bwd_delta_kernel<64><<<nb, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(o),
                                              static_cast<const __nv_bfloat16*>(dout), delta,
                                              qrows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
  // outputs: boxes of 32 rows x 64 columns in the 128-byte swizzle; dQ at
  // d = 64 goes out as 32 x 32 halves without swizzle
  if (!make_tmap_bf16_3d(&tq, q, d, Nq, BH, 64, kTile) ||
      !make_tmap_bf16_3d(&tk, k, d, Nk, BH, 64, kTile) ||
      !make_tmap_bf16_3d(&tv, v, d, Nk, BH, 64, kTile) ||
      !make_tmap_bf16_3d(&tdo, dout, d, Nq, BH, 64, kTile) ||
      !make_tmap_bf16_3d(&tdk, dk, d, Nk, BH, 64, 32) ||
      !make_tmap_bf16_3d(&tdv, dv, d, Nk, BH, 64, 32) ||
      !(d == 128 ? make_tmap_bf16_3d(&tdq, dq, d, Nq, BH, 64, 32)
                 : make_tmap_bf16_3d(&tdq, dq, d, Nq, BH, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE))) {
    *tmap_ok = false;
    return cudaSuccess;
  }
  Params p;
  p.B = B;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.causal = causal ? 1 : 0;
  p.n_qt = (Nq + kTile - 1) / kTile;
  p.n_kt = (Nk + kTile - 1) / kTile;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.key_len = key_len;
  p.lse = lse;
  p.delta = delta;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  void* errp = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&errp, g_bwd_err);
  if (e != cudaSuccess) return e;
  p.err = static_cast<unsigned int*>(errp);
  // the shared-memory opt-in is per function and per device
  static std::atomic<unsigned long long> attr_done{0};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(attr_done.load() & bit)) {
    for (const void* fn : {reinterpret_cast<const void*>(bwd_dq_kernel<128>),
                           reinterpret_cast<const void*>(bwd_dkdv_kernel<128>),
                           reinterpret_cast<const void*>(bwd_dq_kernel<64>),
                           reinterpret_cast<const void*>(bwd_dkdv_kernel<64>)}) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSmemBytes));
      if (e != cudaSuccess) return e;
    }
    attr_done.fetch_or(bit);
  }
  if (Nk > 0 && Nq > 0) {
    const unsigned g = static_cast<unsigned>(BH * p.n_kt);
    if (d == 128)
      bwd_dkdv_kernel<128><<<g, kThreads, kSmemBytes, s>>>(tq, tk, tv, tdo, tdk, tdv, p);
    else
      bwd_dkdv_kernel<64><<<g, kThreads, kSmemBytes, s>>>(tq, tk, tv, tdo, tdk, tdv, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  } else if (Nk > 0) {  // no query: dK = dV = 0
    e = cudaMemsetAsync(dk, 0, static_cast<size_t>(BH) * Nk * d * 2, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, static_cast<size_t>(BH) * Nk * d * 2, s);
    if (e != cudaSuccess) return e;
  }
  if (Nq > 0) {
    if (Nk > 0) {
      const unsigned g = static_cast<unsigned>(BH * p.n_qt);
      if (d == 128)
        bwd_dq_kernel<128><<<g, kThreads, kSmemBytes, s>>>(tq, tk, tv, tdo, tdq, p);
      else
        bwd_dq_kernel<64><<<g, kThreads, kSmemBytes, s>>>(tq, tk, tv, tdo, tdq, p);
      e = cudaGetLastError();
    } else {  // no key: dQ = 0
      e = cudaMemsetAsync(dq, 0, static_cast<size_t>(BH) * Nq * d * 2, s);
    }
  }
  return e;
}

cudaError_t read_and_clear_bwd_error(uint32_t* word) {
  unsigned int w = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&w, bwd::g_bwd_err, sizeof(w));
  if (e != cudaSuccess) return e;
  if (w != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(bwd::g_bwd_err, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
  }
  *word = w;
  return cudaSuccess;
}

}  // namespace osm
