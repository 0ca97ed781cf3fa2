// attn_fwd.cu — exact softmax attention forward on sm_103a tensor cores.
//
// The method: "Online softmax" (zerotofrontier.app), section "Blocks, the
// bridge to FlashAttention": hold a block of query rows, stream key/value
// blocks past it, form the block of scores with a matrix product, summarise it
// per row and merge that summary into the running one (running max m, running
// sum l, unnormalised output O~), rescaling the old state by 2^(m_old - m_new)
// when the max grows; divide once at the end and keep lse = m + log l
// (section "From weights to outputs").  Masks are applied inside the tile loop
// ("Online softmax", guide.dupenodi.dev, "Walking through it"); fully masked
// rows get the merge identity's finalisation (output 0, lse -inf).  Base-2
// exponentials with log2(e) folded into the scale ("Precision, and what can
// still go wrong").
//
// GB300 mapping (one CTA per SM, persistent over work items):
//   work item  = (b, h, pair of 128-row query tiles); both tiles share every
//                streamed K/V tile, and alternate on the tensor core so one
//                tile's softmax overlaps the other tile's matrix products.
//   warp 0     TMA producer: Q tiles once per item (and an L2 prefetch of the
//              next item's Q as soon as its number is known), then K_j together with
//              V_{j-1} (the two tiles step j reads) into one of two pairs of
//              shared-memory slots (128-byte swizzle) under one mbarrier, so
//              each key step costs the MMA thread one wait and one release.
//   warp 1     MMA issuer: per key step j and query tile t,
//              O~_t += P_t V_{j-1} (P_t read straight from TMEM), then
//              S_t = Q_t K_j^T into TMEM over the columns P_t occupied (the
//              tensor pipe runs them in issue order).  The whole warp runs
//              the loop and one elected lane issues each MMA: the descriptor
//              arithmetic then stays warp-uniform, which keeps the issue rate
//              above the tensor pipe's even with two softmax warps competing
//              for the same sub-partition (a single-lane issuer fell below it).
//   warps 4-7  softmax for query tile 0; warps 8-11 for tile 1.  One thread
//              per query row, a rolled loop over the tile's columns in
//              64-column chunks (32 in the normalised form, for registers; no
//              register spills): the chunk
//              TMEM -> registers, mask, scale and subtract the reference in
//              packed f32x2, independent exp2 (so the MUFU latency is
//              covered), row sum, bf16 pack, store P over the S columns
//              already consumed; epilogue: the row's O~ in one TMEM load
//              (which frees the region for the next item at once),
//              O = O~ / l in bf16 through a per-warp shared-memory stage
//              that the tensor-memory engine stores (bulk tensor stores of
//              32 x 64 boxes), lse.  A warp takes its next work item before
//              it waits for O, so the queue and key_len reads stay off the
//              next item's first tile.
//   TMEM       512 columns: S_0 | S_1 | O~_0 | O~_1 (128 fp32 columns each).
// The reference subtracted before exp2 need not be the running maximum: every
// identity of the recurrence holds for any common reference ("Precision, and
// what can still go wrong", second point: any bound on the scores will do).
// So only a row's first tile looks for the maximum (or none, when the caller
// knows a bound and the row starts there).  After that the reference moves by
// whole binades when a chunk would otherwise hold a term above 2^16 (raise:
// everything formed so far is scaled by an exact power of two) or when all of a
// row's terms so far underflow (lower), and to a chunk's exact maximum when
// that chunk outweighs everything before it in the row: a row's dominant term
// then has weight exactly 1, which its bf16 rounding for the P V product leaves
// unchanged, so a nearly one-hot row returns its value's bf16 bits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace osm {
namespace attn {

using namespace ptx;

constexpr int kRows = 128;   // query rows per tile (MMA M)
constexpr int kKeys = 128;   // keys per K/V tile (MMA N of QK^T, K of PV)
constexpr int kSlots = 4;    // K/V ring slots, one 32 KB tile each
constexpr int kPairs = kSlots / 2;  // the ring as (K_j, V_{j-1}) pairs under one barrier
constexpr int kItemSlots = 4;  // depth of the CTA's queue of work-item numbers
constexpr uint32_t kTileBytes = kRows * 128 * 2;  // 32768: a tile slot holds d = 128
constexpr uint32_t kBoxBytes = 128 * 64 * 2;           // one TMA box: 64 columns x 128 rows
constexpr int kThreads = 384;
// A 32-term chunk whose sum stays at or below kSumLimit has no term above it
// (all terms are >= 0), so every P is at most 2^16 times the reference's term.
constexpr float kSumLimit = 65536.0f;
// The most a dominant chunk may lower a caller's bound (binades), so that the
// scale 2^k applied to what the row has accumulated stays finite in FP32.
constexpr float kMaxLower = 120.0f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t kSmemQ = 0;
constexpr uint32_t kSmemKV = 2 * kTileBytes;
constexpr uint32_t kSmemBar = kSmemKV + kSlots * kTileBytes;
enum Bar : uint32_t {
  Q_FULL = 0,       // [2]
  Q_EMPTY = 2,
  KV_FULL = 3,      // [kSlots]
  KV_EMPTY = 3 + kSlots,
  S_FULL = 3 + 2 * kSlots,   // [2]
  P_FULL = S_FULL + 2,       // [2]
  O_FULL = P_FULL + 2,       // [2]
  O_EMPTY = O_FULL + 2,      // [2]
  DRAIN = O_EMPTY + 2,
  ITEM_FULL = DRAIN + 1,     // [kItemSlots]
  ITEM_EMPTY = ITEM_FULL + kItemSlots,  // [kItemSlots]
  NUM_BARS = ITEM_EMPTY + kItemSlots
};
constexpr uint32_t kSmemTmemSlot = kSmemBar + 8 * NUM_BARS;
constexpr uint32_t kSmemAbort = kSmemTmemSlot + 4;
constexpr uint32_t kSmemItems = kSmemAbort + 4;  // int[kItemSlots]: the CTA's item queue
// per softmax warp: a 64-column half of its 32 output rows (bf16, 128 bytes
// a row, in the 128-byte swizzle of the output's tensor map), 1024-aligned
constexpr uint32_t kStageBytes = 32 * 128;
constexpr uint32_t kSmemStage = (kSmemItems + 4 * kItemSlots + 1023) / 1024 * 1024;
constexpr uint32_t kSmemBytes = kSmemStage + 8 * kStageBytes + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
// readers of the item queue: the MMA thread and the eight softmax warps
constexpr uint32_t kItemReaders = 1 + 8;

// TMEM columns
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 256;

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false);  // Q, K both K-major

// error-word sites (kernel id 1 in the top byte); index checks of an
// OSM_CHECKED build use 0x0E01xxxx
constexpr unsigned kSite = 0x01000000u;
constexpr unsigned kChk = 0x0E010000u;


// Bring a 3-D tile into L2 ahead of its load (no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

struct Params {
  int B, H, Nq, Nk;
  int causal;
  int npairs;
  int num_items;
  float scale_log2;
  float m_init;  // starting reference of every row, base-2 units of the scaled scores
  const int32_t* key_len;
  __nv_bfloat16* o;
  float* lse;
  unsigned int* err;
  // work-item counter: the launch's tag in the low 32 bits, the count of
  // items handed out in the high 32 bits (zero at launch)
  unsigned long long* next_item;
  unsigned int tag;
};

struct Item {
  int bh, q0, n_kv, kv_len;
};

__device__ __forceinline__ Item item_info(const Params& p, int item) {
  Item it;
  const int within = item % p.npairs;
  it.bh = item / p.npairs;
  const int pair = p.causal ? (p.npairs - 1 - within) : within;  // causal: longest first
  it.q0 = pair * 2 * kRows;
  const int b = it.bh / p.H;
  int L = p.key_len ? p.key_len[b] : p.Nk;
  L = L < 0 ? 0 : (L > p.Nk ? p.Nk : L);
  it.kv_len = L;
  int end = L;
  if (p.causal) {
    const int last_row = min(it.q0 + 2 * kRows - 1, p.Nq - 1);
    end = min(L, max(0, last_row + 1 + (p.Nk - p.Nq)));
  }
  it.n_kv = (end + kKeys - 1) / kKeys;
  return it;
}

__device__ unsigned int g_err_word;
// Work-item counters.  Each launch takes the next entry (round robin) and
// resets it on its own stream first to (count 0, its own tag), so launches on
// different streams only share a counter when more than kCounters of them are
// in flight at once -- and then the older one finds a foreign tag when it
// next draws an item, records kConflictSite and stops drawing: its output is
// wrong, but osm_device_status reports it.  Launches captured into a CUDA
// graph keep their entry (and tag) for every replay, so they draw from a
// second range that direct launches never use.
constexpr int kCounters = 1024;
__device__ unsigned long long g_item_counter[2 * kCounters];
constexpr unsigned kConflictSite = 0x0C000001u;

// kBounded: every row starts from the caller's bound (p.m_init finite), so no
// tile looks for the maximum and an all-underflow start can lower the reference.
// D: the head dimension, 64 or 128 (a 64-column tile uses half of each slot and
// half of each O~ region; the softmax is the same).
// kNorm: the normalised form of the recurrence ("Online softmax",
// zerotofrontier.app, "From weights to outputs", the second way to write it):
// the output accumulator holds o = O~ / l after every key step.  Each tile's P
// is divided by the new l and the accumulator scaled by l_old / l_new before
// the P V product adds to it; the epilogue divides nothing.  Built to measure
// what the per-step division costs against the single division at the end.
template <bool kBounded, int D, bool kNorm = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + kSmemQ, sKV = sbase + kSmemKV;
  auto bar = [&](uint32_t i) { return sbase + kSmemBar + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemAbort);
  volatile int* item_q = reinterpret_cast<volatile int*>(smem + kSmemItems);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemTmemSlot);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(Q_FULL + t), 1);
      mbar_init(bar(S_FULL + t), 1);
      mbar_init(bar(P_FULL + t), 4);
      mbar_init(bar(O_FULL + t), 1);
      mbar_init(bar(O_EMPTY + t), 4);
    }
    mbar_init(bar(Q_EMPTY), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(KV_FULL + s), 1);
      mbar_init(bar(KV_EMPTY + s), 1);
    }
    mbar_init(bar(DRAIN), 1);
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(bar(ITEM_FULL + s), 1);
      mbar_init(bar(ITEM_EMPTY + s), kItemReaders);
    }
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

  // bounded waits: by one thread, or by a whole warp that then agrees on the outcome
  auto wait_one = [&](uint32_t b, uint32_t parity, unsigned site) -> bool {
    return wait_bounded(b, parity, abort_flag, p.err, site);
  };
  auto wait_all = [&](uint32_t b, uint32_t parity, unsigned site) -> bool {
    return __all_sync(0xffffffffu, wait_bounded(b, parity, abort_flag, p.err, site));
  };
  // Work items are handed out dynamically: the producer thread takes the next
  // item number from a global counter and passes it to the other roles through
  // a small queue in shared memory, so every role of the CTA walks the same
  // item sequence.  -1 ends the sequence.
  uint32_t iq_slot = 0, iq_ph = 0;
  auto iq_advance = [&]() {
    if (++iq_slot == kItemSlots) { iq_slot = 0; iq_ph ^= 1; }
  };

  if (warp < 4) {
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------ TMA producer
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      uint32_t slot = 0, ph = 0, qe_ph = 0;
      uint32_t fill_mask = 0, fill_ph = 0;
      int q_fill = -1;
      int loaded = 0;
      bool ok = true;
      auto publish = [&](int item) -> bool {
        if (!checked(item >= -1 && item < p.num_items, p.err, kChk | 1)) item = -1;
        if (!wait_one(bar(ITEM_EMPTY + iq_slot), iq_ph ^ 1, kSite | 9)) return false;
        item_q[iq_slot] = item;
        mbar_arrive(bar(ITEM_FULL + iq_slot));
        iq_advance();
        return true;
      };
      // Take a ticket: the counter's count, if its tag is this launch's; a
      // foreign tag ends this CTA's items (see g_item_counter).
      auto draw = [&]() -> unsigned int {
        const unsigned long long old = atomicAdd(p.next_item, 1ull << 32);
        if (static_cast<unsigned int>(old) != p.tag) {
          atomicCAS(p.err, 0u, kConflictSite);
          return 0x7fffffffu;
        }
        return static_cast<unsigned int>(old >> 32);
      };
      // the first item of every CTA is its own index (grid <= items); the
      // rest come from the counter, one item ahead of the one being loaded
      int item = blockIdx.x;
      ok = publish(item);
      while (ok && item >= 0) {
        const Item it = item_info(p, item);
        bool published = false;
        unsigned int ticket = 0;
        auto publish_next = [&]() -> bool {
          published = true;
          const int64_t nx = static_cast<int64_t>(gridDim.x) + ticket;
          item = nx < p.num_items ? static_cast<int>(nx) : -1;
          if (item >= 0) {  // the next item's Q into L2 while this one runs
            const Item nit = item_info(p, item);
            if (nit.n_kv > 0)
              for (int t = 0; t < 2 && nit.q0 + t * kRows < p.Nq; ++t)
                for (int c = 0; c < D / 64; ++c)
                  tma_prefetch_l2_3d(&tm_q, c * 64, nit.q0 + t * kRows, nit.bh);
          }
          return publish(item);
        };
        if (it.n_kv > 0) {
          // the copies' coordinates (out-of-range rows read zeros, so these
          // only record a fault): the head and the last key tile
          checked(it.bh < p.B * p.H && (it.n_kv - 1) * kKeys < p.Nk, p.err, kChk | 2);
          if (loaded > 0) {
            if (!(ok = wait_one(bar(Q_EMPTY), qe_ph, kSite | 1))) break;
            qe_ph ^= 1;
          }
          for (int t = 0; t < 2; ++t) {
            mbar_arrive_expect_tx(bar(Q_FULL + t), kRows * D * 2);
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(sQ + t * kTileBytes + c * kBoxBytes, &tm_q, bar(Q_FULL + t), c * 64,
                          it.q0 + t * kRows, it.bh);
          }
          q_fill = loaded & 1;
          ++loaded;
          // the counter's reply is first needed after this item's first K/V copies
          ticket = draw();
          // pair e of the item: K_e (e < n) and V_{e-1} (e > 0), one barrier
          for (int e = 0; ok && e <= it.n_kv; ++e) {
            if (!(ok = wait_one(bar(KV_EMPTY + slot), ph ^ 1, kSite | 2))) break;
            const uint32_t bytes =
                (e < it.n_kv ? kKeys * D * 2u : 0u) + (e > 0 ? kKeys * D * 2u : 0u);
            mbar_arrive_expect_tx(bar(KV_FULL + slot), bytes);
            if (e < it.n_kv)
              for (int c = 0; c < D / 64; ++c)
                tma_load_3d(sKV + (2 * slot) * kTileBytes + c * kBoxBytes, &tm_k,
                            bar(KV_FULL + slot), c * 64, e * kKeys, it.bh);
            if (e > 0)
              for (int c = 0; c < D / 64; ++c)
                tma_load_3d(sKV + (2 * slot + 1) * kTileBytes + c * kBoxBytes, &tm_v,
                            bar(KV_FULL + slot), c * 64, (e - 1) * kKeys, it.bh);
            fill_mask |= 1u << slot;
            fill_ph = (fill_ph & ~(1u << slot)) | (ph << slot);
            if (++slot == kPairs) {
              slot = 0;
              ph ^= 1;
            }
            if (ok && !published) ok = publish_next();
          }
        } else {
          ticket = draw();
        }
        if (ok && !published) ok = publish_next();
      }
      if (!ok) {  // let every copy this thread started land before the CTA exits
        for (int s = 0; s < kPairs; ++s)
          if (fill_mask >> s & 1u) wait_drain(bar(KV_FULL + s), fill_ph >> s & 1u, 200000000ull);
        if (q_fill >= 0)
          for (int t = 0; t < 2; ++t) wait_drain(bar(Q_FULL + t), q_fill, 200000000ull);
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs this loop (so its descriptor arithmetic stays
      // warp-uniform); one elected lane issues each MMA and commit.
      uint32_t slot = 0, ph = 0, qf_ph = 0;
      uint32_t pf_ph[2] = {0, 0}, oe_ph[2] = {0, 0};
      int done = 0;
      bool ok = true;
      const uint64_t dK = sdesc_sw128(0, 16, 1024);     // K-major template (address added)
      const uint64_t dV = sdesc_sw128(0, 16384, 1024);  // MN-major template
      auto commit = [&](uint32_t b) {
        if (elect_one()) mma_commit(b);
        __syncwarp();
      };
      while (ok) {
        if (!(ok = wait_all(bar(ITEM_FULL + iq_slot), iq_ph, kSite | 10))) break;
        const int item = item_q[iq_slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(ITEM_EMPTY + iq_slot));
        iq_advance();
        if (item < 0) break;
        const Item it = item_info(p, item);
        if (it.n_kv == 0) continue;
        for (int t = 0; t < 2 && ok; ++t) ok = wait_all(bar(Q_FULL + t), qf_ph, kSite | 3);
        if (!ok) break;
        qf_ph ^= 1;
        tc_fence_after();
        bool first_pv[2] = {true, true};
        uint32_t v_buf = 0;  // shared-memory address of the V tile of the current pair
        // O~_t += P_t V_{j-1} once the softmax of tile t has stored P_t
        auto issue_pv = [&](int t) -> bool {
          const uint64_t vdesc = dV + (v_buf >> 4);
          if (!wait_all(bar(P_FULL + t), pf_ph[t], kSite | 5)) return false;
          if (first_pv[t] && done > 0) {
            if (!wait_all(bar(O_EMPTY + t), oe_ph[t], kSite | 6)) return false;
            oe_ph[t] ^= 1;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk) {  // 16 keys = 8 TMEM columns of P, 2 KB of V
            if (elect_one())
              mma_ts(tbase + kTmemO + t * 128, tbase + kTmemS + t * 128 + kk * 8,
                     vdesc + ((kk * 2048) >> 4), idesc_bf16_f32(128, D, true),
                     (!first_pv[t] || kk > 0) ? 1u : 0u);
            __syncwarp();
          }
          pf_ph[t] ^= 1;
          first_pv[t] = false;
          return true;
        };
        for (int j = 0; ok && j < it.n_kv; ++j) {
          const uint32_t ps = slot;  // pair j: K_j and (j > 0) V_{j-1}
          if (!(ok = wait_all(bar(KV_FULL + ps), ph, kSite | 4))) break;
          if (++slot == kPairs) { slot = 0; ph ^= 1; }
          tc_fence_after();
          const uint64_t kdesc = dK + ((sKV + (2 * ps) * kTileBytes) >> 4);
          v_buf = sKV + (2 * ps + 1) * kTileBytes;
          for (int t = 0; t < 2 && ok; ++t) {
            if (j > 0 && !(ok = issue_pv(t))) break;
            const uint64_t qdesc = dK + ((sQ + t * kTileBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {  // 16 columns of d = 32 B of a row
              const uint32_t off = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
              if (elect_one())
                mma_ss(tbase + kTmemS + t * 128, qdesc + off, kdesc + off, kIdescS,
                       kk > 0 ? 1u : 0u);
              __syncwarp();
            }
            commit(bar(S_FULL + t));
          }
          if (!ok) break;
          commit(bar(KV_EMPTY + ps));  // pair j read: S(j) and P V_{j-1} issued
          if (j == it.n_kv - 1) commit(bar(Q_EMPTY));
        }
        if (!ok) break;
        const uint32_t ps = slot;  // the item's last pair: V_{n-1}
        if (!(ok = wait_all(bar(KV_FULL + ps), ph, kSite | 4))) break;
        if (++slot == kPairs) { slot = 0; ph ^= 1; }
        tc_fence_after();
        v_buf = sKV + (2 * ps + 1) * kTileBytes;
        for (int t = 0; t < 2 && ok; ++t) {
          if (!(ok = issue_pv(t))) break;
          commit(bar(O_FULL + t));
        }
        if (!ok) break;
        commit(bar(KV_EMPTY + ps));
        ++done;
      }
      if (!ok) {  // wait for every MMA already issued before TMEM is released
        commit(bar(DRAIN));
        if (lane == 0) wait_drain(bar(DRAIN), 0, 200000000ull);
        __syncwarp();
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(32 * wq) << 16;
    const uint32_t tS = tbase + lane_off + kTmemS + t * 128;
    const uint32_t tO = tbase + lane_off + kTmemO + t * 128;
    const float sl2 = p.scale_log2;
    uint32_t sf_ph = 0, of_ph = 0;
    bool ok = true;
    // The next work item from the CTA's queue (-1: none left, -2: the bounded
    // wait gave up) and what it covers.  A warp takes it before it waits for
    // the current item's output, so that the wait and the epilogue, not the
    // next item's first tile, absorb the queue and key_len reads.
    Item nit{};
    auto take_item = [&]() -> int {
      if (!wait_all(bar(ITEM_FULL + iq_slot), iq_ph, kSite | 11)) return -2;
      const int item = item_q[iq_slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(ITEM_EMPTY + iq_slot));
      iq_advance();
      if (item >= 0) nit = item_info(p, item);
      return item;
    };
    int next = take_item();
    while (next >= 0) {
      const Item it = nit;
      const int row = it.q0 + t * kRows + 32 * wq + lane;
      const bool row_ok = row < p.Nq;
      const int64_t orow = static_cast<int64_t>(it.bh) * p.Nq + row;
      const int64_t n_rows = static_cast<int64_t>(p.B) * p.H * p.Nq;
      if (it.n_kv == 0) {
        if (row_ok && checked(orow < n_rows, p.err, kChk | 3)) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + orow * D);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
          p.lse[orow] = kNegInf;
        }
        next = take_item();
        continue;
      }
      int limit = it.kv_len;
      if (p.causal) limit = min(limit, row + 1 + (p.Nk - p.Nq));
      // Every row starts from the reference p.m_init (base-2 units): -inf, so
      // that a row's first tile takes its maximum, or a bound the caller
      // knows.  Later tiles form their terms against the current reference
      // without looking for the maximum: a chunk with a term that may exceed
      // kSumLimit raises the reference, a chunk that outweighs the row so far
      // moves it to the chunk's maximum, and a chunk whose terms all
      // underflow while nothing has accumulated yet lowers it.
      // l: the row's sum of FP32 terms (it gives the lse); lrun: the same sum up
      // to the current chunk (decides which chunk dominates the row); corr
      // (known bound only): the bf16 rounding of the first tile's terms, which
      // start at the caller's bound rather than at a maximum -- O is divided by
      // l + corr, so those terms weigh O exactly as the tensor core used them.
      float m_ref = kBounded ? p.m_init : kNegInf, l = 0.f, lrun = 0.f, corr = 0.f;
      bool at_bound = kBounded;  // the reference is still the caller's bound
      for (int j = 0; j < it.n_kv; ++j) {
        ok = wait_all(bar(S_FULL + t), sf_ph, kSite | 7);
        if (!ok) break;
        sf_ph ^= 1;
        tc_fence_after();
        const int k0 = j * kKeys;
        const bool masked_tile = __any_sync(0xffffffffu, k0 + kKeys > limit);
        const bool first = !kBounded && __any_sync(0xffffffffu, m_ref == kNegInf);
        if (first) {
          float mx[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
#pragma unroll 1
          for (int ch = 0; ch < 4; ++ch) {  // 32 columns at a time: a small register peak
            uint32_t sr[32];
            tmem_ld_x32(tS + 32 * ch, sr);
            if (masked_tile) {
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (k0 + 32 * ch + c >= limit) sr[c] = __float_as_uint(kNegInf);
            }
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
              mx[0] = max3(mx[0], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
              mx[1] = max3(mx[1], __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
              mx[2] = max3(mx[2], __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
              mx[3] = max3(mx[3], __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
            }
          }
          const float m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
          const float m_new = fmaxf(m_ref, m_tile);
          float alpha = 1.f;
          bool resc = false;
          if (m_ref == kNegInf) {
            m_ref = m_new;
          } else if (m_new > m_ref) {  // the tile's maximum becomes the reference exactly
            alpha = ex2(m_ref - m_new);
            l *= alpha;
            lrun *= alpha;
            m_ref = m_new;
            resc = true;
          }
          if (!kNorm && __any_sync(0xffffffffu, resc)) {  // o = O~ / l needs no rescale
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t orr[32];
              tmem_ld_x32(tO + 32 * c, orr);
#pragma unroll
              for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
              tmem_st_x32(tO + 32 * c, orr);
            }
          }
        }
        float nref = (m_ref == kNegInf) ? 0.f : -m_ref;
        // pass over kNch chunks of kCw columns (S read from TMEM), each chunk
        // two-phase: all scale/subtracts, then kCw independent exp2, then the
        // sums and bf16 packs -- so the MUFU latency is covered
        constexpr int kCw = kNorm ? 32 : 64;
        constexpr int kNch = kKeys / kCw;
        float la[4] = {0.f, 0.f, 0.f, 0.f};
        // a chunk whose sum passes thr moves the reference (see below)
        float thr = j > 0 ? fminf(lrun, kSumLimit) : kSumLimit;
#pragma unroll 1
        for (int ch = 0; ch < kNch; ++ch) {
          uint32_t v[kCw], pk[kCw / 2];
          float cs[4];
          auto load_chunk = [&]() {
            tmem_ld_cols(tS + kCw * ch, v);
            if (masked_tile) {
#pragma unroll
              for (int e = 0; e < kCw; ++e)
                if (k0 + kCw * ch + e >= limit) v[e] = __float_as_uint(kNegInf);
            }
          };
          auto exp_chunk = [&]() {
            float pv[kCw];
#pragma unroll
            for (int i = 0; i < kCw / 2; ++i)
              fma2(pv[2 * i], pv[2 * i + 1], __uint_as_float(v[2 * i]),
                   __uint_as_float(v[2 * i + 1]), sl2, sl2, nref, nref);
#pragma unroll
            for (int e = 0; e < kCw; ++e) pv[e] = ex2(pv[e]);
            cs[0] = cs[1] = cs[2] = cs[3] = 0.f;
#pragma unroll
            for (int i = 0; i < kCw / 2; ++i) {
              add2(cs[2 * (i & 1)], cs[2 * (i & 1) + 1], pv[2 * i], pv[2 * i + 1]);
              __nv_bfloat162 h2 = __floats2bfloat162_rn(pv[2 * i], pv[2 * i + 1]);
              pk[i] = *reinterpret_cast<uint32_t*>(&h2);
            }
          };
          load_chunk();
          exp_chunk();
          float csum = (cs[0] + cs[1]) + (cs[2] + cs[3]);
          if (!first) {
            // Three reasons to move the reference.  over: a term may exceed
            // kSumLimit.  dom: the chunk outweighs everything before it in the
            // row, so it may hold the row's dominant term -- that term gets an
            // exact reference (its weight becomes exactly 1, which bf16
            // represents, so O is not off by that weight's rounding).  under
            // (caller's bound only): every term so far underflowed.  Over and
            // dom are one comparison against thr (NaN fails it as well).
            bool any = !(csum <= thr);
            if constexpr (kBounded) any = any || (csum == 0.f && lrun == 0.f);
            if (__any_sync(0xffffffffu, any)) {
              const bool over = !(csum <= kSumLimit);
              const bool dom = j > 0 && csum > lrun;
              const bool under = kBounded && csum == 0.f && lrun == 0.f;
              // The chunk's scores are still in TMEM (P of earlier chunks lies
              // in lower columns): read them again.
              load_chunk();
              float mc = kNegInf;
#pragma unroll
              for (int e = 0; e < kCw; ++e) mc = fmaxf(mc, __uint_as_float(v[e]));
              float m_new = m_ref, alpha = 1.f;
              if (mc != kNegInf) {
                const float mx = mc * sl2;  // the chunk's maximum, base-2 units
                if (dom && (mx > m_ref || (kBounded && at_bound))) {
                  // exact reference: everything formed so far is scaled by
                  // 2^(m_ref - mx), l, O~ and the stored P alike
                  m_new = kBounded ? fmaxf(mx, m_ref - kMaxLower) : mx;
                  if (lrun > 0.f) alpha = ex2(m_ref - m_new);
                  at_bound = false;
                } else if (over || under) {
                  // a whole number k of binades, so that the chunk's largest
                  // term is at most 1: raising (k > 0) scales everything formed
                  // so far by 2^-k, exactly; lowering (caller's bound only)
                  // happens while nothing has accumulated
                  float kr = ceilf(fmaf(mc, sl2, nref));
                  if constexpr (!kBounded) kr = fmaxf(kr, 0.f);
                  m_new = m_ref + kr;
                  // 2^-k exactly; k >= 127 leaves nothing representable (flush to 0)
                  alpha = (kBounded && kr <= 0.f)
                              ? 1.f
                              : (kr >= 127.f ? 0.f : __int_as_float((127 - static_cast<int>(kr)) << 23));
                }
              }
              m_ref = m_new;
              nref = -m_ref;
              l *= alpha;
              lrun *= alpha;
              corr *= alpha;
#pragma unroll
              for (int i = 0; i < 4; ++i) la[i] *= alpha;
              tmem_wait_st();
#pragma unroll 1
              for (int c2 = 0; c2 < ch; ++c2) {  // P of the earlier chunks
                uint32_t pp[kCw / 2];
                tmem_ld_cols(tS + (kCw / 2) * c2, pp);
#pragma unroll
                for (int e = 0; e < kCw / 2; ++e) {
                  const float f0 = __uint_as_float(pp[e] << 16) * alpha;
                  const float f1 = __uint_as_float(pp[e] & 0xffff0000u) * alpha;
                  __nv_bfloat162 h2 = __floats2bfloat162_rn(f0, f1);
                  pp[e] = *reinterpret_cast<uint32_t*>(&h2);
                }
                tmem_st_cols_nowait(tS + (kCw / 2) * c2, pp);
                tmem_wait_st();
              }
              // O~'s last update (P V of the previous tile) completed before S
              // (before a row's first P V it holds no value: scaling it is
              // harmless); o = O~ / l is not scaled
              if constexpr (!kNorm) {
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                  uint32_t orr[32];
                  tmem_ld_x32(tO + 32 * c, orr);
#pragma unroll
                  for (int e = 0; e < 32; ++e)
                    orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                  tmem_st_x32(tO + 32 * c, orr);
                }
              }
              exp_chunk();
              csum = (cs[0] + cs[1]) + (cs[2] + cs[3]);
            }
          }
          lrun += csum;
          thr = j > 0 ? fminf(lrun, kSumLimit) : kSumLimit;  // for the next chunk
          if constexpr (kBounded) {
            if (j == 0) {  // the first tile's terms as rounded to bf16
              float h0 = 0.f, h1 = 0.f;
#pragma unroll
              for (int i = 0; i < kCw / 2; ++i)
                add2(h0, h1, __uint_as_float(pk[i] << 16), __uint_as_float(pk[i] & 0xffff0000u));
              corr += (h0 + h1) - csum;
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) la[i] += cs[i];
          tmem_st_cols_nowait(tS + (kCw / 2) * ch, pk);
        }
        tmem_wait_st();
        if constexpr (kNorm) {
          // o_new = (l_old o + P V) / l_new: P times 1 / l_new (the stored bf16
          // pairs, rounded again), o times l_old / l_new.  The previous P V has
          // completed (it was issued before this tile's S).
          const float l_new = l + ((la[0] + la[1]) + (la[2] + la[3]));
          const float inv = l_new > 0.f ? 1.f / l_new : 0.f;
          const float fo = l * inv;
#pragma unroll 1
          for (int c = 0; c < kKeys / 64; ++c) {
            uint32_t pp[32];
            tmem_ld_x32(tS + 32 * c, pp);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(pp[e] << 16) * inv,
                                                        __uint_as_float(pp[e] & 0xffff0000u) * inv);
              pp[e] = *reinterpret_cast<uint32_t*>(&h2);
            }
            tmem_st_x32(tS + 32 * c, pp);
          }
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t orr[32];
            tmem_ld_x32(tO + 32 * c, orr);
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * fo);
            tmem_st_x32(tO + 32 * c, orr);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(P_FULL + t));
        }
        l += (la[0] + la[1]) + (la[2] + la[3]);
      }
      if (!ok) break;
      next = take_item();
      ok = wait_all(bar(O_FULL + t), of_ph, kSite | 8);
      if (!ok) break;
      of_ph ^= 1;
      tc_fence_after();
      const float inv = kNorm ? (l > 0.f ? 1.f : 0.f) : (l + corr > 0.f ? 1.f / (l + corr) : 0.f);
      // O = O~ / l in bf16, a 64-column half at a time: each thread puts its
      // row's 128 bytes into the warp's stage (32 rows x 128 bytes, 16-byte
      // pieces in the 128-byte swizzle, so the lanes' writes meet no bank
      // twice), and one lane hands the 32 x 64 box to the tensor-memory engine
      // as a bulk store (rows past Nq are not written), so the warp does not
      // wait for its global stores.  (The stage is formed from the shared
      // array itself, so its writes are shared-memory stores.)
      uint8_t* stage = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u) + kSmemStage +
                       (warp - 4) * kStageBytes;
      const uint32_t stage_s = smem_u32(stage);
      uint4* srow = reinterpret_cast<uint4*>(stage + 128 * lane);
      const int row0 = row - lane;  // the warp's first row in its head
      // the row's whole O~ in one TMEM load, so the region is free for the
      // next item's products before the conversions and stores
      uint32_t orr[D];
      tmem_ld_row<D>(tO, orr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(O_EMPTY + t));
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        uint32_t pk2[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(orr[64 * h + 2 * e]) * inv,
                                                    __uint_as_float(orr[64 * h + 2 * e + 1]) * inv);
          pk2[e] = *reinterpret_cast<uint32_t*>(&h2);
        }
        if (lane == 0) bulk_wait_read_0();  // the previous box has left the stage
        __syncwarp();
#pragma unroll
        for (int e = 0; e < 8; ++e)
          srow[e ^ (lane & 7)] = make_uint4(pk2[4 * e], pk2[4 * e + 1], pk2[4 * e + 2], pk2[4 * e + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        // (a warp whose rows all lie past Nq stores nothing)
        if (lane == 0 && row0 < p.Nq && checked(it.bh < p.B * p.H && row0 >= 0, p.err, kChk | 4))
          tma_store_3d(&tm_o, stage_s, 64 * h, row0, it.bh);
      }
      if (row_ok && checked(orow < n_rows, p.err, kChk | 5))
        p.lse[orow] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : kNegInf;
    }
  }

  if (warp >= 4 && lane == 0) bulk_wait_all();  // the epilogue's bulk stores have completed
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// arrives at.  The wait gives up after its time limit, records `site` in the
// error word and returns; the kernel then exits normally.
__global__ void bounded_wait_selftest_kernel(unsigned int* err, unsigned int site) {
  __shared__ __align__(8) uint64_t mbar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  const uint32_t b = smem_u32(&mbar);
  mbar_init(b, 1);
  fence_mbar_init();
  wait_bounded(b, 0, reinterpret_cast<volatile int*>(&abort_flag), err, site);
}

// every query row fully masked (no key at all): O = 0, lse = -inf
__global__ void attn_empty_kernel(__nv_bfloat16* o, float* lse, int64_t rows, int d) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < rows * (d / 8)) reinterpret_cast<uint4*>(o)[i] = make_uint4(0, 0, 0, 0);
  if (i < rows) lse[i] = kNegInf;
}

}  // namespace attn

int sm_count_current_device() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

cudaError_t launch_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int H, int Nq, int Nk, int d, float scale, int causal,
                            const int32_t* key_len, float score_bound, bool normalised,
                            cudaStream_t s, bool* tmap_ok) {
  using namespace attn;
  *tmap_ok = true;
  const int64_t rows = static_cast<int64_t>(B) * H * Nq;
  if (Nk == 0) {
    const int64_t n = rows * (d / 8);
    attn_empty_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(
        static_cast<__nv_bfloat16*>(o), lse, rows, d);
    return cudaGetLastError();
  }
  CUtensorMap tq, tk, tv, to;
  const uint64_t BH = static_cast<uint64_t>(B) * H;
  if (!make_tmap_bf16_3d(&tq, q, d, Nq, BH, 64, kRows) ||
      !make_tmap_bf16_3d(&tk, k, d, Nk, BH, 64, kKeys) ||
      !make_tmap_bf16_3d(&tv, v, d, Nk, BH, 64, kKeys) ||
      !make_tmap_bf16_3d(&to, o, d, Nq, BH, 64, 32)) {
    *tmap_ok = false;
    return cudaSuccess;
  }
  Params p;
  p.B = B;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.causal = causal ? 1 : 0;
  p.npairs = (Nq + 2 * kRows - 1) / (2 * kRows);
  const int64_t items = static_cast<int64_t>(BH) * p.npairs;
  p.num_items = static_cast<int>(items);
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  // a known bound on the scaled scores starts every row there; without one a
  // row's first tile takes its maximum
  p.m_init = std::isfinite(score_bound)
                 ? static_cast<float>(static_cast<double>(score_bound) * 1.4426950408889634)
                 : kNegInf;
  p.key_len = key_len;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  void* errp = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&errp, g_err_word);
  if (e != cudaSuccess) return e;
  p.err = static_cast<unsigned int*>(errp);
  void* ctrp = nullptr;
  e = cudaGetSymbolAddress(&ctrp, g_item_counter);
  if (e != cudaSuccess) return e;
  static std::atomic<unsigned int> next_direct{0}, next_captured{0};
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(s, &cap);
  if (e != cudaSuccess) return e;
  const unsigned int seq =
      cap == cudaStreamCaptureStatusNone ? next_direct.fetch_add(1) : next_captured.fetch_add(1);
  const unsigned int slot = (cap == cudaStreamCaptureStatusNone ? 0 : kCounters) + seq % kCounters;
  p.next_item = static_cast<unsigned long long*>(ctrp) + slot;
  p.tag = seq;
  // reset: tag in the low word, count 0 in the high word
  auto memset32 = memset_d32_fn();
  if (!memset32) return cudaErrorNotSupported;
  if (memset32(reinterpret_cast<CUdeviceptr>(p.next_item), p.tag, 1, s) != CUDA_SUCCESS)
    return cudaErrorUnknown;
  e = cudaMemsetAsync(reinterpret_cast<unsigned int*>(p.next_item) + 1, 0, sizeof(unsigned int), s);
  if (e != cudaSuccess) return e;
  // the shared-memory opt-in is per function and per device
  static std::atomic<unsigned long long> attr_done{0};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(attr_done.load() & bit)) {
    for (const void* fn : {reinterpret_cast<const void*>(attn_fwd_kernel<false, 128>),
                           reinterpret_cast<const void*>(attn_fwd_kernel<true, 128>),
                           reinterpret_cast<const void*>(attn_fwd_kernel<false, 64>),
                           reinterpret_cast<const void*>(attn_fwd_kernel<true, 64>),
                           reinterpret_cast<const void*>(attn_fwd_kernel<false, 128, true>),
                           reinterpret_cast<const void*>(attn_fwd_kernel<false, 64, true>)}) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSmemBytes));
      if (e != cudaSuccess) return e;
    }
    attr_done.fetch_or(bit);
  }
  const int grid = static_cast<int>(items < sm_count_current_device() ? items
                                                                      : sm_count_current_device());
  const bool bounded = std::isfinite(score_bound);
  if (normalised) {
    if (d == 128)
      attn_fwd_kernel<false, 128, true><<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, to, p);
    else
      attn_fwd_kernel<false, 64, true><<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, to, p);
  } else if (d == 128) {
    if (bounded)
      attn_fwd_kernel<true, 128><<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, to, p);
    else
      attn_fwd_kernel<false, 128><<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, to, p);
  } else {
    if (bounded)
      attn_fwd_kernel<true, 64><<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, to, p);
    else
      attn_fwd_kernel<false, 64><<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, to, p);
  }
  return cudaGetLastError();
}

cudaError_t launch_bounded_wait_selftest(cudaStream_t s) {
  void* errp = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&errp, attn::g_err_word);
  if (e != cudaSuccess) return e;
  attn::bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(static_cast<unsigned int*>(errp),
                                                      0x7f0000a1u);
  return cudaGetLastError();
}

cudaError_t read_and_clear_device_error(cudaStream_t s, uint32_t* word) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  unsigned int w = 0;
  e = cudaMemcpyFromSymbol(&w, attn::g_err_word, sizeof(w));
  if (e != cudaSuccess) return e;
  if (w != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(attn::g_err_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
  }
  *word = w;
  return cudaSuccess;
}

}  // namespace osm
