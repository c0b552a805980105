// Forward attention for head dimension 256 on sm_103a (tcgen05, TMA, TMEM).
//
// The method is the same as the d = 64 / 128 kernel (FlashAttention-2, Alg. 1:
// S = Q K^T tile by tile, online softmax with a lazily rescaled O, P never
// leaving the SM, O / l and the row log-sum-exp at the end), with the same
// masks (causal aligned to the end of the keys, sliding window with sink keys,
// varlen sequences, "TileLang tutorial, ch.15", sections 3.4 and 5.3) and the
// same logit sink (section 4.6).  What changes is the budget: two 128-row Q
// tiles would need 2 x (128 + 256) tensor-memory columns, more than 512, so a
// CTA takes one Q tile and spends the columns on two S buffers and O:
//
//   tensor memory  S[0] [0,128)  S[1] [128,256)  O [256,512)
//   shared memory  Q (4 atoms of 128 rows x 64 columns, 64 KB), K (4 atoms),
//                  V (4 atoms), barriers: 192 KB + 1 KB
//
// The grid is persistent: one CTA per SM walks its share of the Q tiles
// (items dealt in bands of gridDim.x, every other band in reverse order),
// and every role's barrier phases run on over the CTA's whole sequence of
// key tiles.  Q, like K, is released atom by atom after the last S of an
// item, so the next item's Q and K stream in while that S still runs.
//
// Warps: 0-3 softmax (thread r owns query row q0 + r, lanes of its quarter of
// tensor memory), 4 TMA producer, 5 MMA issuer.  Per key tile n the issuer
// runs S(n+1) = Q K(n+1)^T into the other S buffer, then O += P(n) V(n) as soon
// as the softmax has written P(n) (bf16 pairs over the first 64 columns of
// S(n)'s buffer): the softmax of one tile overlaps the products of the next.
// K is released atom by atom (each atom feeds four of the sixteen K-steps of
// S), so K(n+1) streams in while S(n) is still running; V is released once
// O += P V has read it.  O += P V is one N = 256 product per K-step.
//
// Keys in a paged cache (the kPaged instantiation, query blocks packed as for
// varlen): every 128-key tile is eight 16-token pages looked up in the
// sequence's page-table row, each atom of the tile loaded as eight 16-row
// boxes from the 4-D map over the page pool (a 16-row box at a 2 KB offset
// keeps the 128-byte swizzle phase of the atom).
#include "attn_internal.h"
#include "sm103_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

namespace attn {
namespace {

using namespace ptx;

constexpr int kR = 128;                 // query rows per CTA, keys per key tile
constexpr int kD = 256;                 // head dimension
constexpr int kAtom = 128 * 128;        // one 128-row x 64-column bf16 atom (16 KB)
constexpr int kNAtom = kD / 64;         // atoms per tile
constexpr int kThr = 192;               // warps 0-3 softmax, 4 producer, 5 MMA issuer
constexpr int kWarpProducer = 4;
constexpr int kWarpIssuer = 5;
constexpr int kOffQ = 0;
constexpr int kOffK = kNAtom * kAtom;
constexpr int kOffV = 2 * kNAtom * kAtom;
constexpr int kOffBar = 3 * kNAtom * kAtom;
// q_full[4], q_empty[4], k_full[4], k_empty[4], v_full, v_empty, s_full[2],
// p_ready[2], o_done[2], drain, and the tensor-memory address slot
constexpr int kNumBars = 4 * kNAtom + 1 + 1 + 2 + 2 + 2 + 1;
constexpr int kSmem = kOffBar + (kNumBars + 1) * 8 + 1024;
static_assert(kSmem <= 227 * 1024, "shared memory");
constexpr uint32_t kColO = 2 * kR;
// O is rescaled only when the running maximum has grown by more than 2^8 in
// the exponent since the value the exponentials are taken against (the
// partial sums stay far from overflow, and the final O / l is unchanged).
constexpr float kRescaleLog2 = 8.0f;
constexpr int kNoLowerBound = -(1 << 29);
constexpr int kPage = 16;                // keys per page of a paged cache
constexpr int kPagesPerTile = kR / kPage;

struct P256 {
  __nv_bfloat16* o;
  float* lse;
  const float* sink;  // logit sink per query head, or null
  const int* cu_q;    // varlen sequence starts, or null (dense)
  const int* cu_k;
  const int* page_table;  // paged keys: [B, max_pages] physical pages
  const int* seqlens_k;   // paged keys: key count of every sequence [B]
  int max_pages, num_pages;
  long long o_sb, o_ss, o_sh;  // O strides (elements): batch, row, head
  int o_v8;                    // every O row starts on 32 bytes: 32-byte stores
  int B, Hq, Hkv, Sq, Skv, total_q, num_qt, num_items;
  float scale, scale2;
  int causal, window, n_sink;
  uint64_t wait_limit_ns;
  int* status;
};

// One CTA's Q tile: coordinates, lengths, and the visible-key bounds of its
// first and last row (key k is visible to row q iff k <= hi(q) and, with a
// window, k > lo(q) or k < n_sink).
struct Tile {
  int bseq, h, hk, q0, Lq, Lk, off, q_base, k_base, b_coord;
  int hi_min, hi_max, lo_min, lo_max;
  int jlo, jhi, sinkT, n_act;
};

// Item order: without a causal mask the Q tiles of one (sequence, head) are
// adjacent so that they read the same K and V through L2; with one, the
// last (longest) Q tiles of every head come first.
template <bool kPaged>
__device__ __forceinline__ bool decode_tile(const P256& p, int item, Tile& w, bool report) {
  const int per = p.Hq * p.B;
  int x = item, qt;
  if (kPaged) {
    // Query blocks against a paged cache read far more keys than they have
    // queries: the items that share a sequence's key head (its query tiles
    // and the query heads of the group) are adjacent, so that the CTAs
    // running together read its keys and values once from HBM (taking the
    // query tiles longest first across all heads instead re-read them 3.5x).
    const int G = p.Hq / p.Hkv;
    const int hg = x % G;
    x /= G;
    qt = p.num_qt - 1 - x % p.num_qt;
    x /= p.num_qt;
    w.h = (x % p.Hkv) * G + hg;
    w.bseq = x / p.Hkv;
  } else if (p.causal) {
    qt = p.num_qt - 1 - x / per;
    x %= per;
    w.h = x % p.Hq;
    w.bseq = x / p.Hq;
  } else {
    qt = x % p.num_qt;
    x /= p.num_qt;
    w.h = x % p.Hq;
    w.bseq = x / p.Hq;
  }
  if (kPaged) {
    // Packed queries against a paged cache: the sequence's keys are its
    // first seqlens_k[b] cache slots.
    const int a = p.cu_q[w.bseq], e = p.cu_q[w.bseq + 1];
    const int lk = p.seqlens_k[w.bseq];
    if (a < 0 || e < a || e > p.total_q || e - a > p.Sq || lk < 0 ||
        lk > p.max_pages * kPage) {
      if (report) atomicOr(p.status, kStatusBadInput);
      return false;
    }
    w.Lq = e - a;
    w.Lk = lk;
    w.q_base = a;
    w.k_base = 0;
    w.b_coord = 0;
  } else if (p.cu_q != nullptr) {
    const int a = p.cu_q[w.bseq], e = p.cu_q[w.bseq + 1];
    const int ka = p.cu_k[w.bseq], ke = p.cu_k[w.bseq + 1];
    if (a < 0 || e < a || e > p.total_q || ka < 0 || ke < ka || e - a > p.Sq) {
      if (report) atomicOr(p.status, kStatusBadInput);
      return false;
    }
    w.Lq = e - a;
    w.Lk = ke - ka;
    w.q_base = a;
    w.k_base = ka;
    w.b_coord = 0;
  } else {
    w.Lq = p.Sq;
    w.Lk = p.Skv;
    w.q_base = 0;
    w.k_base = 0;
    w.b_coord = w.bseq;
  }
  w.q0 = qt * kR;
  if (w.q0 >= w.Lq) return false;
  w.off = w.Lk - w.Lq;
  w.hk = w.h / (p.Hq / p.Hkv);
  const int last = min(w.q0 + kR, w.Lq) - 1;
  w.hi_min = p.causal ? min(w.q0 + w.off, w.Lk - 1) : w.Lk - 1;
  w.hi_max = p.causal ? min(last + w.off, w.Lk - 1) : w.Lk - 1;
  w.lo_min = p.window > 0 ? w.q0 + w.off - p.window : kNoLowerBound;
  w.lo_max = p.window > 0 ? last + w.off - p.window : kNoLowerBound;
  // Active key tiles: j <= jhi and (j >= jlo or j < sinkT).
  w.sinkT = p.window > 0 ? (p.n_sink + kR - 1) / kR : 0;
  if (w.hi_max < 0 || w.Lk <= 0) {
    w.jlo = 0;
    w.jhi = -1;
    w.n_act = 0;
    return true;
  }
  w.jhi = w.hi_max / kR;
  if (p.window <= 0)
    w.jlo = 0;
  else if (w.lo_min >= w.Lk - 1)
    w.jlo = w.jhi + 1;  // only sink keys are visible
  else
    w.jlo = w.lo_min < 0 ? 0 : (w.lo_min + 1) / kR;
  const int ns = min(w.sinkT, w.jhi + 1);
  w.n_act = ns + max(0, w.jhi - max(w.jlo, w.sinkT) + 1);
  return true;
}

// The n-th item of this CTA, or -1 past the last: bands of gridDim.x items,
// every other band dealt in reverse CTA order.
__device__ __forceinline__ int item_at(int n, int num_items) {
  const int G = gridDim.x;
  const int pos = (n & 1) ? (G - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  const long long k = static_cast<long long>(n) * G + pos;
  return k < num_items ? static_cast<int>(k) : -1;
}

// The n-th active key tile (sink tiles first, then the window's range).
__device__ __forceinline__ int tile_at(const Tile& w, int n) {
  const int ns = min(w.sinkT, w.jhi + 1);
  return n < ns ? n : max(w.jlo, w.sinkT) + (n - ns);
}

// Does every row of the Q tile see every key of key tile j?
__device__ __forceinline__ bool interior(const Tile& w, int j, int window, int n_sink) {
  const int ka = j * kR, kb = ka + kR - 1;
  if (kb > w.hi_min) return false;
  if (window > 0 && !(ka > w.lo_max || kb < n_sink)) return false;
  return true;
}

__device__ __forceinline__ void reg_fence256(uint32_t& r) { asm volatile("" : "+r"(r)); }

__device__ __forceinline__ void tmem_wait_ld256() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void fail256(int* status, volatile int* abort_flag) {
  atomicOr(status, kStatusTimeout);
  *abort_flag = 1;
}

// Bounded wait by the whole warp (every lane tests; the result is uniform).
__device__ __forceinline__ bool wwait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                      const P256& p) {
  const bool ok =
      __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.wait_limit_ns));
  if (!ok && (threadIdx.x & 31) == 0) fail256(p.status, abort_flag);
  return ok;
}

template <bool kPaged>
__global__ void __launch_bounds__(kThr, 1)
    attn_fwd256_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const P256 p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars;                   // [4] Q atom a of the current item landed
  uint64_t* q_empty = q_full + kNAtom;       // [4] the item's last S has read Q atom a
  uint64_t* k_full = q_empty + kNAtom;       // [4] K atom a of the current key tile landed
  uint64_t* k_empty = k_full + kNAtom;       // [4] S has read K atom a
  uint64_t* v_full = k_empty + kNAtom;       // V tile landed
  uint64_t* v_empty = v_full + 1;            // O += P V has read V
  uint64_t* s_full = v_empty + 1;            // [2] S of a key tile is in tensor memory
  uint64_t* p_ready = s_full + 2;            // [2] P written (128 arrivals)
  uint64_t* o_done = p_ready + 2;            // [2] O += P V of an even / odd key tile done
  uint64_t* drain = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  __shared__ int abort_s;
  volatile int* abort_flag = &abort_s;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int a = 0; a < kNAtom; ++a) {
      mbar_init(&q_full[a], 1);
      mbar_init(&q_empty[a], 1);
      mbar_init(&k_full[a], 1);
      mbar_init(&k_empty[a], 1);
    }
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_ready[b], kR);
      mbar_init(&o_done[b], 1);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
    abort_s = 0;
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // Counters over the CTA's whole sequence: key tiles (one S, one P V each)
  // and items with key tiles (one Q load each).  Items without a visible key
  // (n_act = 0) only have an epilogue.
  if (warp == kWarpProducer) {
    // ============================================================ TMA producer
    int k_cnt[kNAtom] = {0, 0, 0, 0};  // loads issued into each K atom
    int v_loads = 0;                   // V tiles whose loads were issued
    int q_loads = 0;                   // items whose Q was loaded
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int item = item_at(it, p.num_items);
      if (item < 0) break;
      Tile w;
      if (!decode_tile<kPaged>(p, item, w, lane == 0) || w.n_act == 0) continue;
      const int N = w.n_act;
      // Paged cache: the physical page of rows 16 pp.. of key tile j, for
      // lane pp (pages past the sequence's last are replaced by that last
      // page, whose rows are masked; an index outside the pool is reported
      // and page 0 read instead).
      // Each tile's pages are read from the page table two tiles ahead of
      // its loads (lookup) and checked when used (checked); the K and V
      // loads of a tile share them.
      auto lookup = [&](int n) -> int {
        int phys = 0;
        if (kPaged && n < N && lane < kPagesPerTile) {
          const int np = (w.Lk + kPage - 1) / kPage;
          const int lp = min(tile_at(w, n) * kPagesPerTile + lane, np - 1);
          phys = p.page_table[static_cast<size_t>(w.bseq) * p.max_pages + lp];
        }
        return phys;
      };
      auto checked = [&](int phys) -> int {
        if (kPaged && lane < kPagesPerTile && (phys < 0 || phys >= p.num_pages)) {
          atomicOr(p.status, kStatusBadInput);
          phys = 0;
        }
        return phys;
      };
      // One 64-column atom of key tile j into dst (expected bytes: one atom).
      auto load_atom = [&](const CUtensorMap* map, uint8_t* dst, uint64_t* bar, int a, int j,
                           int phys) {
        if constexpr (kPaged) {
          // lane pp issues the box of its own page: one warp instruction
          // starts the copies of all eight pages of the atom
          if (lane < kPagesPerTile)
            tma_load_4d(dst + lane * kPage * 128, map, bar, a * 64, w.hk, 0, phys);
          __syncwarp();
        } else {
          (void)phys;
          tma_load_4d_w(dst, map, bar, a * 64, w.hk, w.k_base + j * kR, w.b_coord);
        }
      };
      // Key tile n of the item; for n = 0 the item's Q atoms go first, each
      // once the previous item's last S has read it.
      auto load_k = [&](int n, int phys) {
        const int j = tile_at(w, n);
        for (int a = 0; a < kNAtom; ++a) {
          if (n == 0) {
            if (q_loads > 0 && !wwait(&q_empty[a], (q_loads - 1) & 1, abort_flag, p))
              return false;
            mbar_arrive_expect_tx_w(&q_full[a], kAtom);
            tma_load_4d_w(sQ + a * kAtom, &tmQ, &q_full[a], a * 64, w.h, w.q_base + w.q0,
                          w.b_coord);
          }
          // atom a is free once the S before has read it
          if (k_cnt[a] > 0 && !wwait(&k_empty[a], (k_cnt[a] - 1) & 1, abort_flag, p))
            return false;
          mbar_arrive_expect_tx_w(&k_full[a], kAtom);
          load_atom(&tmK, sK + a * kAtom, &k_full[a], a, j, phys);
          ++k_cnt[a];
        }
        if (n == 0) ++q_loads;
        return true;
      };
      int ph0 = checked(lookup(0));  // pages of tile n (V(n) still to load)
      int ph1 = lookup(1);            // tile n + 1, in flight
      ok = load_k(0, ph0);
      for (int n = 0; ok && n < N; ++n) {
        // K runs one key tile ahead of V: K(n + 1) as S(n) releases its atoms,
        // V(n) once the P V before has read the V before.
        const int ph2 = lookup(n + 2);
        if (n + 1 < N) {
          ph1 = checked(ph1);
          if (!load_k(n + 1, ph1)) {
            ok = false;
            break;
          }
        }
        if (v_loads > 0 && !wwait(v_empty, (v_loads - 1) & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        const int j = tile_at(w, n);
        const int phys = ph0;
        mbar_arrive_expect_tx_w(v_full, kNAtom * kAtom);
#pragma unroll
        for (int a = 0; a < kNAtom; ++a) load_atom(&tmV, sV + a * kAtom, v_full, a, j, phys);
        ++v_loads;
        ph0 = ph1;
        ph1 = ph2;
      }
    }
    // Every copy issued lands before the CTA can leave (a load is issued
    // only after the previous one into the same buffer has been consumed,
    // so waiting for the last phase of each barrier covers them all).
    for (int a = 0; a < kNAtom; ++a) {
      if (q_loads > 0) mbar_wait(&q_full[a], (q_loads - 1) & 1, nullptr, p.wait_limit_ns);
      if (k_cnt[a] > 0) mbar_wait(&k_full[a], (k_cnt[a] - 1) & 1, nullptr, p.wait_limit_ns);
    }
    if (v_loads > 0) mbar_wait(v_full, (v_loads - 1) & 1, nullptr, p.wait_limit_ns);
  } else if (warp == kWarpIssuer) {
    // ============================================================ MMA issuer
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, kR, false);
    constexpr uint32_t idesc_o = idesc_bf16_f32(128, kD, true);
    const uint64_t dq = sdesc_sw128(smem_addr(sQ), 16, 1024);
    const uint64_t dk = sdesc_sw128(smem_addr(sK), 16, 1024);
    const uint64_t dv = sdesc_sw128(smem_addr(sV), kAtom, 1024);
    int g = 0;   // key tiles of earlier items
    int qi = 0;  // items with key tiles before this one
    // S of key tile g + n = Q K^T into buffer (g + n) % 2: K-steps 4a .. 4a+3
    // read atom a of Q and K; atom a of K is released as soon as its four
    // steps are done, and after the item's last S atom a of Q too.
    auto issue_s = [&](int n, bool last) -> bool {
      const int t = g + n;
      const uint32_t tS = tmem + (t & 1) * kR;
#pragma unroll 1
      for (int a = 0; a < kNAtom; ++a) {
        if ((n == 0 && !wwait(&q_full[a], qi & 1, abort_flag, p)) ||
            !wwait(&k_full[a], t & 1, abort_flag, p))
          return false;
        tc_fence_after_sync();
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
          const uint64_t ko = static_cast<uint64_t>((a * kAtom + s4 * 32) >> 4);
          mma_bf16_ss_w(tS, dq + ko, dk + ko, idesc_s, (a > 0 || s4 > 0) ? 1u : 0u);
        }
        mma_commit_w(&k_empty[a]);
        if (last) mma_commit_w(&q_empty[a]);
      }
      mma_commit_w(&s_full[t & 1]);
      return true;
    };
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int item = item_at(it, p.num_items);
      if (item < 0) break;
      Tile w;
      if (!decode_tile<kPaged>(p, item, w, false) || w.n_act == 0) continue;
      const int N = w.n_act;
      ok = issue_s(0, N == 1);
      for (int n = 0; ok && n < N; ++n) {
        if (n + 1 < N && !issue_s(n + 1, n + 2 == N)) {
          ok = false;
          break;
        }
        // O += P V of key tile t: A = P (bf16 pairs, key-step kk at column
        // 8 kk of S(t)'s buffer), B = V read along d (N = 256, one product
        // per step).  The item's first overwrites O: the epilogue before it
        // has read O out before the p_ready arrival waited for here.
        const int t = g + n;
        if (!wwait(&p_ready[t & 1], (t >> 1) & 1, abort_flag, p) ||
            !wwait(v_full, t & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t tP = tmem + (t & 1) * kR;
#pragma unroll
        for (int kk = 0; kk < kR / 16; ++kk)
          mma_bf16_ts_w(tmem + kColO, tP + 8 * kk, dv + kk * (2048 >> 4), idesc_o,
                        (n > 0 || kk > 0) ? 1u : 0u);
        mma_commit_w(v_empty);
        mma_commit_w(&o_done[t & 1]);
      }
      g += N;
      ++qi;
    }
    // Every product issued has completed before tensor memory is released.
    mma_commit_w(drain);
    mbar_wait(drain, 0, nullptr, p.wait_limit_ns);
  } else if (warp < 4) {
    // ============================================================ softmax warps 0-3
    const int r = warp * 32 + lane;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    int g = 0;  // key tiles of earlier items
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int item = item_at(it, p.num_items);
      if (item < 0) break;
      Tile w;
      if (!decode_tile<kPaged>(p, item, w, false)) continue;
      const int N = w.n_act;
      const int q = w.q0 + r;  // sequence-relative query row
      const bool valid = q < w.Lq;
      const int hi = p.causal ? min(q + w.off, w.Lk - 1) : w.Lk - 1;
      const int lo = p.window > 0 ? q + w.off - p.window : kNoLowerBound;
      float m_run = -INFINITY;   // running maximum of the raw scores
      float m_used = -INFINITY;  // maximum the exponentials are taken against
      float l = 0.f;             // sum of the exponentials (against m_used)
      // O is formed from bf16-rounded P while l sums the fp32 values; when one
      // key dominates a row that rounding error does not cancel, so the
      // difference p - bf16(p) of every tile's largest p is taken out of the
      // normaliser of O (not of the log-sum-exp).
      float corr = 0.f;
      for (int n = 0; n < N; ++n) {
        const int j = tile_at(w, n);
        const int t = g + n;
        if (!wwait(&s_full[t & 1], (t >> 1) & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t tS = taddr + (t & 1) * kR;
        uint32_t s[kR];
#pragma unroll
        for (int c = 0; c < kR / 32; ++c) tmem_ld_x32(tS + 32 * c, s + 32 * c);
        tmem_wait_ld256();
#pragma unroll
        for (int e = 0; e < kR; ++e) reg_fence256(s[e]);
        if (!interior(w, j, p.window, p.n_sink)) {
          // key k = j*128 + c is visible iff k <= hi and (k > lo or k < n_sink)
          const int ka = j * kR;
#pragma unroll
          for (int c = 0; c < kR; ++c) {
            const int k = ka + c;
            if (!(k <= hi && (k > lo || k < p.n_sink))) s[c] = __float_as_uint(-INFINITY);
          }
        }
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = __uint_as_float(s[e]);
#pragma unroll
        for (int c = 8; c < kR; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], __uint_as_float(s[c]));
        const float tmax = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                 fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        m_run = fmaxf(m_run, tmax);
        // Lazy rescale: move the reference maximum only when the scores have
        // outgrown it by 2^8; O (already holding earlier tiles) is then scaled
        // by 2^((m_used - m_run) scale2) once O += P V of the previous tile is
        // done.  The tensor-memory accesses are warp-collective: a warp
        // rescales if any of its rows must (the others multiply by 1).
        const bool first = (m_used == -INFINITY);
        const bool grow =
            first ? (m_run != -INFINITY) : ((m_run - m_used) * p.scale2 > kRescaleLog2);
        const bool resc = grow && !first;
        if (__any_sync(0xffffffffu, resc)) {
          if (!wwait(&o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, abort_flag, p)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const float alpha = resc ? ex2_approx((m_used - m_run) * p.scale2) : 1.f;
#pragma unroll 1
          for (int c = 0; c < kD / 32; ++c) {
            uint32_t o[32];
            tmem_ld_x32(taddr + kColO + 32 * c, o);
            tmem_wait_ld256();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_x32(taddr + kColO + 32 * c, o);
          }
          tmem_st_wait();
          l *= alpha;
          corr *= alpha;
        }
        if (grow) m_used = m_run;
        // P = 2^(S scale2 - m_used scale2) as bf16 pairs over the first 64
        // columns of the buffer (key-step kk of O += P V at column 8 kk); a
        // row that has seen no key yet has m_used = -inf and every P = 0.
        const float nms = first && !grow ? 0.f : -m_used * p.scale2;
        float sum0 = 0.f, sum1 = 0.f;
        uint32_t pk[kR / 2];
#pragma unroll
        for (int e = 0; e < kR / 2; ++e) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(s[2 * e]), p.scale2, nms));
          const float p1 = ex2_approx(fmaf(__uint_as_float(s[2 * e + 1]), p.scale2, nms));
          if (e & 1)
            sum1 += p0 + p1;
          else
            sum0 += p0 + p1;
          pk[e] = pack_bf16x2(p0, p1);
        }
        l += sum0 + sum1;
        {  // the tile's largest p, with the arithmetic used for it above
          const float ptop = ex2_approx(fmaf(tmax, p.scale2, nms));
          corr += ptop - __uint_as_float(pack_bf16x2(0.f, ptop) & 0xffff0000u);
        }
        tmem_st_x32(tS, pk);
        tmem_st_x32(tS + 32, pk + 32);
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&p_ready[t & 1]);
      }
      if (!ok) break;
      // -------------------------------------------------------------- epilogue
      const bool have_o = N > 0;
      if (have_o) {
        const int t = g + N - 1;
        if (!wwait(&o_done[t & 1], (t >> 1) & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
      }
      g += N;
      // O / l, or with a logit sink sigma of this head one more term of the
      // denominator taken against m* = max(sigma, m scale) ("TileLang
      // tutorial, ch.15", section 4.6); a row that saw no key gets O = 0.
      const bool seen = have_o && l > 0.f;
      const float sg = p.sink ? p.sink[w.h] : -INFINITY;
      float inv, lse_row;
      if (sg == -INFINITY) {
        inv = seen ? 1.f / (l - corr) : 0.f;
        lse_row = seen ? fmaf(m_used, p.scale, logf(l)) : -INFINITY;
      } else {
        const float am = seen ? m_used * p.scale : -INFINITY;
        const float mst = fmaxf(am, sg);
        const float e1 = seen ? expf(am - mst) : 0.f;
        const float e2 = expf(sg - mst);
        inv = e1 / fmaf(l - corr, e1, e2);
        lse_row = mst + logf(fmaf(l, e1, e2));
      }
      const size_t orow =
          (p.cu_q ? static_cast<size_t>(w.q_base + q) * p.o_ss
                  : static_cast<size_t>(w.bseq) * p.o_sb + static_cast<size_t>(q) * p.o_ss) +
          static_cast<size_t>(w.h) * p.o_sh;
#pragma unroll 1
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t o[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
        if (have_o) {
          tmem_ld_x32(taddr + kColO + 32 * c, o);
          tmem_wait_ld256();
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) reg_fence256(o[e]);
        if (valid) {
          uint32_t wv[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            wv[e] = seen ? pack_bf16x2(__uint_as_float(o[2 * e]) * inv,
                                       __uint_as_float(o[2 * e + 1]) * inv)
                         : 0u;
          uint4* dst = reinterpret_cast<uint4*>(p.o + orow + 32 * c);
          if (p.o_v8) {
            st_global_v8(dst, wv);
            st_global_v8(dst + 2, wv + 8);
          } else {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              dst[v4] = make_uint4(wv[4 * v4], wv[4 * v4 + 1], wv[4 * v4 + 2], wv[4 * v4 + 3]);
          }
        }
      }
      if (valid && p.lse != nullptr) {
        const size_t li = p.cu_q ? static_cast<size_t>(w.h) * p.total_q + w.q_base + q
                                 : (static_cast<size_t>(w.bseq) * p.Hq + w.h) * p.Sq + q;
        p.lse[li] = lse_row;
      }
      // The next item's first O += P V waits for this warp's next p_ready
      // arrival, made after the reads of O above.
      tc_fence_before_sync();
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_attn_fwd256(const FwdLaunch& a, cudaStream_t stream) {
  if (a.d != kD) return cudaErrorInvalidValue;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    for (auto fn : {attn_fwd256_kernel<false>, attn_fwd256_kernel<true>}) {
      attr_err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
      if (attr_err != cudaSuccess) return;
    }
  });
  if (attr_err != cudaSuccess) return attr_err;
  P256 p;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.sink = a.sink;
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.page_table = a.page_table;
  p.seqlens_k = a.seqlens_k;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.o_sb = a.o_sb;
  p.o_ss = a.o_ss;
  p.o_sh = a.o_sh;
  p.o_v8 = (reinterpret_cast<uintptr_t>(a.o) % 32 == 0) && a.o_sb % 16 == 0 && a.o_ss % 16 == 0 &&
           a.o_sh % 16 == 0;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Skv = a.Skv;
  p.total_q = a.total_q;
  p.num_qt = (a.Sq + kR - 1) / kR;
  p.scale = a.scale;
  p.scale2 = a.scale * 1.4426950408889634f;
  p.causal = a.causal;
  p.window = a.window;
  p.n_sink = a.n_sink;
  p.wait_limit_ns = kWaitLimitNs;
  p.status = a.status;
  const long long items = static_cast<long long>(p.num_qt) * a.Hq * a.B;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  p.num_items = static_cast<int>(items);
  // Dense calls: persistent, one CTA per SM (each holds all 512 tensor-
  // memory columns), the equal-length items dealt in bands.  Packed and
  // paged calls: one CTA per item, so that the hardware hands the next item
  // to whichever SM frees first (item costs follow the sequence lengths,
  // which a fixed dealing balances badly: 1.54 ms persistent against 1.22 ms
  // on a paged batch of 2,048-8,192 cached keys).
  const bool packed = a.cu_q != nullptr || a.page_table != nullptr;
  const long long grid = packed ? items : std::min<long long>(items, std::max(a.num_sms, 1));
  if (a.page_table != nullptr)
    attn_fwd256_kernel<true><<<static_cast<unsigned>(grid), kThr, kSmem, stream>>>(a.tmQ, a.tmK,
                                                                                  a.tmV, p);
  else
    attn_fwd256_kernel<false><<<static_cast<unsigned>(grid), kThr, kSmem, stream>>>(a.tmQ, a.tmK,
                                                                                   a.tmV, p);
  return cudaGetLastError();
}

}  // namespace attn
