// Backward pass of the dense exact-attention forward on sm_103a: dQ, dK, dV
// for an output gradient dO, from Q, K, V, O and the forward's row LSE.
//
// The pages give no backward formulas ("TileLang tutorial, ch.15
// Operators: Attention", section 5.4 only measures what a bf16, atomically
// accumulated dQ loses); the kernels follow the chain rule through O = P V
// and the row softmax, recomputing P from the saved LSE instead of storing
// it:
//   P  = exp(scale Q K^T - LSE),      dV = P^T dO,
//   dP = dO V^T,   D = rowsum(dO * O) (= rowsum(P * dP)),
//   dS = P * (dP - D),   dQ = scale dS K,   dK = scale dS^T Q.
// Every gradient is accumulated in fp32 in tensor memory over its whole
// reduction and written once, so the results do not depend on scheduling
// (no atomics): dK and dV of a key tile by one CTA, looping over every
// query tile of every query head that reads the key head; dQ of a query tile
// by one CTA, looping over the key tiles.  For dense calls both grids are
// persistent (one CTA per SM walking its share of the tiles, every barrier
// phase carried over from one tile to the next, the next tile's loads and
// first products overlapping the last one's output), for packed calls one
// CTA per tile.
//
// Kernels:
//   attn_bwd_rowstat_kernel  D and LSE in base 2 per query row, padded to
//                            whole 128-row tiles (+inf LSE on pad rows and
//                            on rows that saw no key, so their P is 0);
//   attn_bwd_dkdv_kernel<D>  warps 0-7: S^T -> P^T, dP^T -> dS^T (warps w
//                            and w+4 share key row 32 (w % 4) + lane and
//                            split the 128 query columns in halves); warp 8:
//                            TMA producer (K, V once; Q per query tile in
//                            three slots, dO and the two row vectors in
//                            two); warp 9: MMA issuer.  Tensor memory:
//                            S^T [0,128), dP^T [128,256), dV [256,256+D),
//                            dK [256+D,..).
//   attn_bwd_dq_kernel<D>    the same roles over key tiles for one query
//                            tile (K in three slots, V in two): S [0,128),
//                            released once read out; dP (then dS) in
//                            [128,256) and [384,512) alternately; dQ
//                            [256,256+D).  S and dP of the next tile run
//                            while dS of this one is formed.
// Products (tcgen05, kind::f16, M=128, fp32 in tensor memory):
//   S^T = K Q^T, dP^T = V dO^T   (both operands K-major in shared memory)
//   dV += P^T dO, dK += dS^T Q   (A from tensor memory, B MN-major)
//   S = Q K^T, dP = dO V^T, dQ += dS K.
// P and dS enter the second products as bf16, like P in the forward.
//
// Masks are the forward's: causal aligned to the end of each sequence's keys,
// a sliding window of W keys with n_sink sink keys visible to every query
// that may see them causally, packed (varlen) sequences through cu_seqlens
// ("TileLang tutorial, ch.15", sections 3.4, 5.2 and 5.3).  The dK/dV kernel
// walks the query tiles that see its key tile (one contiguous range: the
// window bounds it above unless the tile holds sink keys); the dQ kernel
// walks the sink tiles, then its window of key tiles.
#include "attn_bwd_common.cuh"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

namespace attn {
namespace {

using namespace ptx;

template <int D>
struct BwdCfg {
  static constexpr int kTile = kB * D * 2;       // one 128 x D bf16 tile
  static constexpr int kAtoms = D / 64;          // 128-byte swizzle atoms per row
  static constexpr int kAtomBytes = kB * 128;    // one atom column of a tile
  static constexpr int kVec = kB * 4;            // one fp32 row vector of a tile
  // dK/dV kernel: K, V resident; Q tiles in three slots (read by S^T early
  // and by dK late in a query tile's products), dO tiles with the tile's two
  // row vectors (-LSE2, -D) in two.  No alignment slack: the kernel checks
  // that the dynamic shared memory starts on 1024 bytes (it does on this GPU,
  // with no static shared memory) and reports otherwise.
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTile;
  static constexpr int kOffQs = 2 * kTile;
  static constexpr int kDSlot = kTile + 2 * kVec;
  static constexpr int kOffDs = kOffQs + 3 * kTile;
  static constexpr int kOffBarKV = kOffDs + 2 * kDSlot;
  static constexpr int kSmemKV = kOffBarKV + 24 * 8;
  static_assert(kDSlot % 1024 == 0, "dO slots on the swizzle atom");
  // dQ kernel: Q, dO resident; K tiles in three slots (read by S early and
  // by dQ late in a key tile's products), V tiles in two (read by dP only)
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kTile;
  static constexpr int kOffKs = 2 * kTile;
  static constexpr int kOffVs = kOffKs + 3 * kTile;
  static constexpr int kOffBarQ = kOffVs + 2 * kTile;
  static constexpr int kSmemQ = kOffBarQ + 24 * 8 + 1024;
  static_assert(kSmemKV <= 227 * 1024 && kSmemQ <= 227 * 1024, "shared memory");
  // Each CTA allocates all 512 tensor-memory columns: ask for enough shared
  // memory that a second CTA never shares the SM (its allocation would wait).
  static constexpr int kOneCta = 116 * 1024;
  static constexpr int kLaunchKV = kSmemKV > kOneCta ? kSmemKV : kOneCta;
  static constexpr int kLaunchQ = kSmemQ > kOneCta ? kSmemQ : kOneCta;
};

// Eight lanes per query row (four rows per warp at a time): D = sum_t dO_t
// O_t (fp32) and LSE2 = LSE log2(e), both stored negated (the kernels add
// them); rows past Sq (to the tile boundary) and rows whose LSE is -inf (no
// key) get -LSE2 = -inf and D = 0, so every P built from them is 0.
template <int D>
__global__ void attn_bwd_rowstat_kernel(BwdParams p) {
  const int lane = threadIdx.x % 32, sub = lane / 8, l8 = lane % 8;
  const long long nrow = static_cast<long long>(p.B) * p.Hq * p.Sqp;
  const long long wstride = static_cast<long long>(gridDim.x) * (blockDim.x / 32) * 4;
  for (long long rw0 = (static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32) * 4;
       rw0 < nrow; rw0 += wstride) {
    const long long rw = rw0 + sub;
    float acc = 0.f, l2 = INFINITY;
    int i = 0;
    bool row_ok = false;
    if (rw < nrow) {
      i = static_cast<int>(rw % p.Sqp);
      const long long bh = rw / p.Sqp;
      const int h = static_cast<int>(bh % p.Hq), b = static_cast<int>(bh / p.Hq);
      SeqGeo g;
      row_ok = seq_geo(p, b, g, i == 0 && h == 0 && l8 == 0) && i < g.Lq;
      if (row_ok) {
        const size_t base = ((static_cast<size_t>(g.q_row0) + i) * p.Hq + h) * D;
        const float l = p.cu_q != nullptr
                            ? p.lse[static_cast<size_t>(h) * p.total_q + g.q_row0 + i]
                            : p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.Sq + i];
        // eight bf16 (16 bytes) per lane and load, every load of the row in
        // flight before the first product
        constexpr int kLd = D / 64;
        uint4 gv[kLd], ov[kLd];
#pragma unroll
        for (int c = 0; c < kLd; ++c) {
          gv[c] = *reinterpret_cast<const uint4*>(p.dout + base + l8 * 8 + c * 64);
          ov[c] = *reinterpret_cast<const uint4*>(p.o + base + l8 * 8 + c * 64);
        }
#pragma unroll
        for (int c = 0; c < kLd; ++c) {
          const uint32_t gw[4] = {gv[c].x, gv[c].y, gv[c].z, gv[c].w};
          const uint32_t ow[4] = {ov[c].x, ov[c].y, ov[c].z, ov[c].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc = fmaf(__uint_as_float(gw[e] << 16), __uint_as_float(ow[e] << 16), acc);
            acc = fmaf(__uint_as_float(gw[e] & 0xffff0000u),
                       __uint_as_float(ow[e] & 0xffff0000u), acc);
          }
        }
        l2 = (l == -INFINITY) ? INFINITY : l * kLog2eB;
      }
    }
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (l8 == 0 && rw < nrow) {
      p.dvec[rw] = row_ok ? -acc : 0.f;  // stored negated: added, not subtracted
      p.lse2[rw] = -l2;
    }
  }
}

// Gradient of the logit sink of query head h (blockIdx.x): with the sink as
// one more softmax column without a value row, dS of that column is
// P_sink (0 - D) per row, so dsink_h = -sum_rows exp(sink_h - LSE) D over the
// rows of the head.  The workspace holds -LSE log2(e) and -D per row (pad
// rows and rows without a key: -inf, 0).  Each thread sums a fixed set of
// rows and the block adds the partial sums in a fixed tree, so the result
// does not depend on scheduling.
constexpr int kSinkThreads = 256;
__global__ void __launch_bounds__(kSinkThreads)
    attn_bwd_dsink_kernel(const float* __restrict__ lse2, const float* __restrict__ dvec,
                          const float* __restrict__ sink, float* __restrict__ dsink, int B, int Hq,
                          int Sqp) {
  __shared__ float part[kSinkThreads];
  const int h = blockIdx.x;
  const float s2 = sink[h] * kLog2eB;  // -inf: no sink, a zero gradient
  float acc = 0.f;
  const long long rows = static_cast<long long>(B) * Sqp;
  for (long long r = threadIdx.x; r < rows; r += kSinkThreads) {
    const long long b = r / Sqp, i = r % Sqp;
    const size_t w = (static_cast<size_t>(b) * Hq + h) * Sqp + i;
    const float x = s2 + lse2[w];
    if (x > -INFINITY) acc = fmaf(exp2f(x), dvec[w], acc);  // P_sink (-D)
  }
  part[threadIdx.x] = acc;
  __syncthreads();
  for (int n = kSinkThreads / 2; n > 0; n >>= 1) {
    if (threadIdx.x < n) part[threadIdx.x] += part[threadIdx.x + n];
    __syncthreads();
  }
  if (threadIdx.x == 0) dsink[h] = part[0];
}


// One key tile of the dK/dV kernel: which, and the query tiles that see it.
struct KvItem {
  int kt, hk, b, k0, qt_lo, nq, ntiles;
  SeqGeo sg;
};

// Item order.  Under a causal mask the key tile is outermost, so that the
// longest (key tile 0 has the most query tiles) come first; without one
// every item is the same work and the key tiles of one (batch, key head) are
// adjacent, so the CTAs running together read the same query and
// output-gradient tiles through L2.  False for a key tile past its
// sequence's keys (nothing to write).
__device__ __forceinline__ bool kv_item(const BwdParams& p, int item, KvItem& it) {
  const int nkt_all = (p.Skv + kB - 1) / kB;
  if (p.causal) {
    it.kt = item / (p.B * p.Hkv);
    it.hk = (item / p.B) % p.Hkv;
    it.b = item % p.B;
  } else {
    it.kt = item % nkt_all;
    it.hk = (item / nkt_all) % p.Hkv;
    it.b = item / (nkt_all * p.Hkv);
  }
  it.k0 = it.kt * kB;
  if (!seq_geo(p, it.b, it.sg, false) || it.k0 >= it.sg.Lk) return false;
  const int nqt = (it.sg.Lq + kB - 1) / kB;
  const int off = it.sg.Lk - it.sg.Lq;
  // The query tiles that see a key of the tile: from the first query that
  // sees key k0 (causal) to the last that sees key k0 + 127 (window; a tile
  // holding sink keys is seen to the end).
  int qt_lo = 0, qt_hi = nqt - 1;
  if (p.causal) {
    const int qmin = it.k0 - off;  // first query that sees key k0
    qt_lo = qmin <= 0 ? 0 : qmin / kB;
  }
  if (p.window > 0 && it.k0 >= p.n_sink) {
    const int qmax = it.k0 + kB - 1 - off + p.window - 1;  // last query that sees key k0 + 127
    qt_hi = qmax < 0 ? -1 : min(qt_hi, qmax / kB);
  }
  it.qt_lo = qt_lo;
  it.nq = qt_hi >= qt_lo ? qt_hi - qt_lo + 1 : 0;
  it.ntiles = (p.Hq / p.Hkv) * it.nq;  // (query head, query tile) pairs, head-major
  return true;
}

// dK and dV of key tiles (128 keys) of a key head: items (key tile, key head,
// batch), the grid persistent for dense calls (one CTA per SM walking its
// items, every barrier phase carried over the CTA's whole sequence of query
// tiles) and one CTA per item for packed ones (item costs follow the
// sequence lengths).
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmDO, BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  chain_allow_next();
  // The layout fills shared memory with no room to round the window up to
  // the swizzle atom: a window off the boundary is reported, not used.
  if (smem_addr(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    chain_join_prev();
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBarKV);
  uint64_t* kv_full = bars;       // K and V tiles landed
  uint64_t* q_full = bars + 1;    // [3] Q of a query tile landed
  uint64_t* q_free = bars + 4;    // [3] S^T and dK of that tile are done
  uint64_t* d_full = bars + 7;    // [2] dO, -LSE2, -D of a query tile landed
  uint64_t* d_free = bars + 9;    // [2] dP^T, dV and dK of that tile are done
  uint64_t* sa_full = bars + 11;  // S^T is in tensor memory
  uint64_t* sb_full = bars + 12;  // dP^T is in tensor memory
  uint64_t* pa_ready = bars + 13; // P^T written (one arrival per compute thread)
  uint64_t* pb_ready = bars + 14; // dS^T written (one arrival per compute thread)
  uint64_t* done = bars + 15;     // every product of the item is done
  uint64_t* drain = bars + 16;
  uint64_t* kv_empty = bars + 17; // the item's last products reading K and V are done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 18);
  // in the layout too: no static shared memory ahead of the window
  int* abort_s = reinterpret_cast<int*>(bars + 19);
  volatile int* abort_flag = abort_s;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = p.Hq / p.Hkv;
  const int num_items = ((p.Skv + kB - 1) / kB) * p.Hkv * p.B;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_free[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&d_full[s], 1);
      mbar_init(&d_free[s], 1);
    }
    mbar_init(sa_full, 1);
    mbar_init(sb_full, 1);
    mbar_init(pa_ready, kComputeThreads);
    mbar_init(pb_ready, kComputeThreads);
    mbar_init(done, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
    *abort_s = 0;
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  auto qslot = [&](int u) { return smem + C::kOffQs + (u % 3) * C::kTile; };   // Q of query tile u
  auto dslot = [&](int u) { return smem + C::kOffDs + (u & 1) * C::kDSlot; };  // dO, vectors of tile u

  // Counters over the CTA's items: query tiles (one Q and one dO load, one
  // set of products each) and items with query tiles (one K / V load each).  Items
  // without a query tile only write zeros.
  if (warp == kWarpProd) {
    // ================================================================ producer
    int kv_loads = 0, issued = 0, q_loads = 0;  // issued: dO loads (and query tiles)
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int item = bwd_item_at(n, num_items);
      if (item < 0) break;
      KvItem it;
      if (!kv_item(p, item, it) || it.ntiles == 0) continue;
      // K and V are single-buffered: the previous item's last S^T and dP^T
      // must be done with them
      if (kv_loads > 0 && !warp_wait(kv_empty, (kv_loads - 1) & 1, abort_flag, p)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx_w(kv_full, 2 * C::kTile);
#pragma unroll
      for (int a = 0; a < C::kAtoms; ++a) {
        tma_load_4d_w(sK + a * C::kAtomBytes, &tmK, kv_full, a * 64, it.hk,
                      it.sg.k_base + it.k0, it.sg.b_coord);
        tma_load_4d_w(sV + a * C::kAtomBytes, &tmV, kv_full, a * 64, it.hk,
                      it.sg.k_base + it.k0, it.sg.b_coord);
      }
      ++kv_loads;
      // Warm L2 with the next item's K and V: they are single-buffered, so
      // their load waits for this item's last products and is then on the
      // way to the next item's first S^T.
      {
        KvItem nx;
        const int nitem = bwd_item_at(n + 1, num_items);
        if (nitem >= 0 && kv_item(p, nitem, nx) && nx.ntiles > 0) {
#pragma unroll
          for (int a = 0; a < C::kAtoms; ++a) {
            tma_prefetch_4d_w(&tmK, a * 64, nx.hk, nx.sg.k_base + nx.k0, nx.sg.b_coord);
            tma_prefetch_4d_w(&tmV, a * 64, nx.hk, nx.sg.k_base + nx.k0, nx.sg.b_coord);
          }
        }
      }
      // Q of query tile u goes to slot u % 3 once S^T and dK of tile u - 3
      // are done, dO and the row vectors to slot u % 2 once tile u - 2 is
      // done: both loads run more than a query tile ahead of their first
      // product.
      for (int t = 0; t < it.ntiles; ++t) {
        const int u = issued;
        const int h = it.hk * G + t / it.nq, qt = it.qt_lo + t % it.nq;
        if (u >= 3 && !warp_wait(&q_free[u % 3], ((u / 3) - 1) & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx_w(&q_full[u % 3], C::kTile);
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a)
          tma_load_4d_w(qslot(u) + a * C::kAtomBytes, &tmQ, &q_full[u % 3], a * 64, h,
                        it.sg.q_base + qt * kB, it.sg.b_coord);
        ++q_loads;
        if (u >= 2 && !warp_wait(&d_free[u & 1], ((u >> 1) - 1) & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        uint8_t* ds = dslot(u);
        mbar_arrive_expect_tx_w(&d_full[u & 1], C::kTile + 2 * C::kVec);
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a)
          tma_load_4d_w(ds + a * C::kAtomBytes, &tmDO, &d_full[u & 1], a * 64, h,
                        it.sg.q_base + qt * kB, it.sg.b_coord);
        const size_t vrow =
            (static_cast<size_t>(it.b) * p.Hq + h) * p.Sqp + static_cast<size_t>(qt) * kB;
        bulk_load_1d_w(ds + C::kTile, p.lse2 + vrow, C::kVec, &d_full[u & 1]);
        bulk_load_1d_w(ds + C::kTile + C::kVec, p.dvec + vrow, C::kVec, &d_full[u & 1]);
        ++issued;
      }
    }
    // Let every copy issued land before the CTA can leave.
    if (kv_loads > 0) warp_wait(kv_full, (kv_loads - 1) & 1, nullptr, p);
    for (int s = 0; s < 3; ++s) {
      const int n_s = (q_loads - s + 2) / 3;  // loads issued into Q slot s
      if (n_s > 0) warp_wait(&q_full[s], (n_s - 1) & 1, nullptr, p);
    }
    for (int s = 0; s < 2; ++s) {
      const int n_s = (issued - s + 1) / 2;  // loads issued into dO slot s
      if (n_s > 0) warp_wait(&d_full[s], (n_s - 1) & 1, nullptr, p);
    }
  } else if (warp == kWarpIssue) {
    // ================================================================ MMA issuer
    // Per query tile t the pipe runs dP^T(t), dV(t), S^T(t+1), dK(t): S^T of
    // the next tile overwrites P^T(t) once dV(t) has read it, while the
    // compute warps form dS^T(t) from P^T kept in their registers; dP^T(t+1)
    // overwrites dS^T(t) once dK(t) has read it.  An item's first dV and dK
    // overwrite the accumulators: they wait for the P^T / dS^T arrivals the
    // compute warps make after reading the previous item's dK and dV out.
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, kB, false);
    constexpr uint32_t idesc_g = idesc_bf16_f32(128, D, true);
    const uint64_t dk = sdesc_sw128(smem_addr(sK), 16, 1024);
    const uint64_t dvk = sdesc_sw128(smem_addr(sV), 16, 1024);
    const uint32_t tS = tmem, tP = tmem + kB, tDV = tmem + 2 * kB, tDK = tmem + 2 * kB + D;
    int T = 0;    // query tiles of earlier items
    int kvi = 0;  // items with query tiles before this one
    auto issue_st = [&](int u) -> bool {  // S^T(u) = K Q(u)^T
      if (!warp_wait(&q_full[u % 3], (u / 3) & 1, abort_flag, p)) return false;
      tc_fence_after_sync();
      const uint64_t dqk = sdesc_sw128(smem_addr(qslot(u)), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t ko = kmajor_step<C::kAtomBytes>(kk);
        mma_bf16_ss_w(tS, dk + ko, dqk + ko, idesc_s, kk > 0 ? 1u : 0u);
      }
      mma_commit_w(sa_full);
      return true;
    };
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int item = bwd_item_at(n, num_items);
      if (item < 0) break;
      KvItem it;
      if (!kv_item(p, item, it) || it.ntiles == 0) continue;
      const int nt = it.ntiles;
      ok = warp_wait(kv_full, kvi & 1, abort_flag, p);
      if (ok) tc_fence_after_sync();
      if (ok) ok = issue_st(T);
      for (int t = 0; ok && t < nt; ++t) {
        const int u = T + t;  // query tile over the CTA's items
        if (!warp_wait(&d_full[u & 1], (u >> 1) & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t dst_ = smem_addr(dslot(u));
        const uint64_t ddok = sdesc_sw128(dst_, 16, 1024);
        // dP^T(t) = V dO(t)^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ko = kmajor_step<C::kAtomBytes>(kk);
          mma_bf16_ss_w(tP, dvk + ko, ddok + ko, idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(sb_full);
        // the item's last products reading K (its last S^T, issued before)
        // and V: the producer may load the next item's K and V
        if (t + 1 == nt) mma_commit_w(kv_empty);
        // dV += P^T dO(t) (A from tensor memory, K = queries; B read along d)
        if (!warp_wait(pa_ready, u & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint64_t dqm = sdesc_sw128(smem_addr(qslot(u)), C::kAtomBytes, 1024);
        const uint64_t ddom = sdesc_sw128(dst_, C::kAtomBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kB / 16; ++kk)
          mma_bf16_ts_w(tDV, tS + packed_col(kk), ddom + kk * (2048 >> 4), idesc_g,
                        (t > 0 || kk > 0) ? 1u : 0u);
        if (t + 1 < nt && !issue_st(u + 1)) {
          ok = false;
          break;
        }
        // dK += dS^T Q(t)
        if (!warp_wait(pb_ready, u & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kB / 16; ++kk)
          mma_bf16_ts_w(tDK, tP + packed_col(kk), dqm + kk * (2048 >> 4), idesc_g,
                        (t > 0 || kk > 0) ? 1u : 0u);
        // the tile's last products: its Q slot, and its dO slot (whose row
        // vectors the compute warps read before publishing dS^T)
        mma_commit_w(&q_free[u % 3]);
        mma_commit_w(&d_free[u & 1]);
      }
      if (ok) mma_commit_w(done);
      T += nt;
      ++kvi;
    }
    // Every product issued has finished before tensor memory is released.
    mma_commit_w(drain);
    warp_wait(drain, 0, nullptr, p);
  } else if (warp < kComputeWarps) {
    // ================================================================ compute warps
    const int wq = warp & 3, wh = warp >> 2;  // lane quarter, column half
    const int r = wq * 32 + lane;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint64_t sc2 = pf2(p.scale2, p.scale2);
    int T = 0;    // query tiles of earlier items
    int kvi = 0;  // items with query tiles before this one
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int item = bwd_item_at(n, num_items);
      if (item < 0) break;
      KvItem it;
      if (!kv_item(p, item, it)) continue;
      const int nt = it.ntiles;
      const int k_idx = it.k0 + r;
      const int off = it.sg.Lk - it.sg.Lq;
      for (int t = 0; t < nt; ++t) {
        const int u = T + t;
        // the row vectors came by bulk copy with dO: observe that barrier too
        if (!warp_wait(sa_full, u & 1, abort_flag, p) ||
            !warp_wait(&d_full[u & 1], (u >> 1) & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const int qt = it.qt_lo + t % it.nq;
        // this warp's 64 entries of the two row vectors (-LSE2, -D)
        const uint32_t nl2_addr = smem_addr(dslot(u) + C::kTile) + 4 * 64 * wh;
        const uint32_t nd2_addr = nl2_addr + 4 * kB;
        // column c (query qt*128 + c) is visible to this key row iff
        // cmin <= c <= cmax: causal from below, the window from above (not for
        // sink keys); key rows past the sequence see nothing
        int cmin = p.causal ? k_idx - off - qt * kB : -(1 << 30);
        int cmax = (p.window > 0 && k_idx >= p.n_sink) ? k_idx - off + p.window - 1 - qt * kB
                                                        : (1 << 30);
        if (k_idx >= it.sg.Lk) cmin = 1 << 30;
        // P^T of this warp's 64 columns: written to tensor memory for dV and
        // kept in registers (bf16 pairs) for dS^T, because S^T of the next
        // tile replaces it.
        uint32_t pkeep[32];
        {
          uint32_t ra[64];
          uint64_t nl2[16];
          tmem_ld_x32(taddr + 64 * wh, ra);
          tmem_ld_x32(taddr + 64 * wh + 32, ra + 32);
          lds_chunk(nl2_addr, nl2);
          tmem_ld_wait_b();
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int c4 = 2 * wh + j;
            float pf[32];
            // x = S scale2 - LSE2 in pairs (the vector holds -LSE2); the mask
            // is applied only to a chunk the diagonal crosses
            if (j == 1) lds_chunk(nl2_addr + 128, nl2);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              reg_fence_b(ra[32 * j + 2 * e]);
              reg_fence_b(ra[32 * j + 2 * e + 1]);
              const uint64_t x2 = pf2_fma(pf2(__uint_as_float(ra[32 * j + 2 * e]),
                                              __uint_as_float(ra[32 * j + 2 * e + 1])),
                                          sc2, nl2[e]);
              float x0, x1;
              pf2_split(x2, x0, x1);
              pf[2 * e] = ex2_approx(x0);
              pf[2 * e + 1] = ex2_approx(x1);
            }
            if (cmin > 32 * c4 || cmax < 32 * c4 + 31) {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (32 * c4 + e < cmin || 32 * c4 + e > cmax) pf[e] = 0.f;
            }
            pack32(pf, pkeep + 16 * j);
            tmem_st_x16(taddr + 64 * wh + 16 * j, pkeep + 16 * j);
          }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(pa_ready);
        // dS^T = P^T (dP^T - D), from the bf16 P^T
        if (!warp_wait(sb_full, u & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        {
          uint32_t ra[64];
          uint64_t nd2[16];  // -D in pairs
          tmem_ld_x32(taddr + kB + 64 * wh, ra);
          tmem_ld_x32(taddr + kB + 64 * wh + 32, ra + 32);
          lds_chunk(nd2_addr, nd2);
          tmem_ld_wait_b();
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float pf[32];
            uint32_t pk[16];
            if (j == 1) lds_chunk(nd2_addr + 128, nd2);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              reg_fence_b(ra[32 * j + 2 * e]);
              reg_fence_b(ra[32 * j + 2 * e + 1]);
              const uint32_t w = pkeep[16 * j + e];
              const uint64_t p2 = pf2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
              const uint64_t g2 = pf2_add(pf2(__uint_as_float(ra[32 * j + 2 * e]),
                                              __uint_as_float(ra[32 * j + 2 * e + 1])),
                                          nd2[e]);
              pf2_split(pf2_mul(p2, g2), pf[2 * e], pf[2 * e + 1]);
            }
            pack32(pf, pk);
            tmem_st_x16(taddr + kB + 64 * wh + 16 * j, pk);
          }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(pb_ready);
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (nt > 0) {
        if (!warp_wait(done, kvi & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
      }
      const bool valid = k_idx < it.sg.Lk;
      const size_t orow = ((static_cast<size_t>(it.sg.k_row0) + k_idx) * p.Hkv + it.hk) * D;
      constexpr int kHalfChunks = D / 64;  // 32-column chunks in a column half
#pragma unroll 1
      for (int g = 0; g < 2; ++g) {  // 0: dV, 1: dK (times scale)
        __nv_bfloat16* dst = (g == 0 ? p.dv : p.dk) + orow;
        const float mul = g == 0 ? 1.f : p.scale;
#pragma unroll 1
        for (int c = wh * kHalfChunks; c < (wh + 1) * kHalfChunks; ++c) {
          uint32_t ra[32];
          if (nt > 0) {
            tmem_ld_x32(taddr + 2 * kB + g * D + 32 * c, ra);
            tmem_ld_wait_b();
          }
          float f[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            reg_fence_b(ra[e]);
            f[e] = nt > 0 ? __uint_as_float(ra[e]) * mul : 0.f;
          }
          uint32_t pk[16];
          pack32(f, pk);
          if (valid) store_row32(dst + 32 * c, pk, p.v8);
        }
      }
      // The next item's first dV and dK wait for this warp's next arrivals,
      // made after the reads of the accumulators above.
      tc_fence_before_sync();
      T += nt;
      if (nt > 0) ++kvi;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 512);
  chain_join_prev();
}

// One query tile of the dQ kernel: which, and the key tiles its rows see.
struct QItem {
  int qt, h, b, hk, q0, jlo, jhi, sinkT, ns, nkt;
  SeqGeo sg;
  // the n-th key tile walked: sink tiles first, then the window's range
  __device__ __forceinline__ int tile_at(int n) const {
    return n < ns ? n : max(jlo, sinkT) + (n - ns);
  }
};

// Item order.  Under a causal mask the query tile is outermost, the last
// (longest) first; without one the query tiles of one (batch, head) are
// adjacent, so the CTAs running together read the same key and value tiles.
// False for a query tile past its sequence's queries (nothing to write).
__device__ __forceinline__ bool q_item(const BwdParams& p, int item, QItem& it) {
  const int nqt_all = p.Sqp / kB;
  if (p.causal) {
    it.qt = nqt_all - 1 - item / (p.B * p.Hq);
    it.h = (item / p.B) % p.Hq;
    it.b = item % p.B;
  } else {
    it.qt = item % nqt_all;
    it.h = (item / nqt_all) % p.Hq;
    it.b = item / (nqt_all * p.Hq);
  }
  it.hk = it.h / (p.Hq / p.Hkv);
  it.q0 = it.qt * kB;
  if (!seq_geo(p, it.b, it.sg, false) || it.q0 >= it.sg.Lq) return false;
  const int off = it.sg.Lk - it.sg.Lq;
  // The key tiles the tile's rows see: the sink tiles, then the window's
  // tiles from the first key above the first row's window bound up to the
  // last key any row sees (causal bound, end of the keys).
  int jhi = (it.sg.Lk - 1) / kB;
  if (p.causal) {
    const int qlast = min(it.q0 + kB - 1, it.sg.Lq - 1);
    const int kmax = min(it.sg.Lk - 1, qlast + off);  // last key any row of the tile sees
    jhi = kmax >= 0 ? kmax / kB : -1;
  }
  if (it.sg.Lk <= 0) jhi = -1;
  int jlo = 0, sinkT = 0;
  if (p.window > 0) {
    const int lo = it.q0 + off - p.window;  // keys above lo are in the first row's window
    jlo = lo < 0 ? 0 : (lo + 1) / kB;
    sinkT = (p.n_sink + kB - 1) / kB;
  }
  it.jlo = jlo;
  it.jhi = jhi;
  it.sinkT = sinkT;
  it.ns = min(sinkT, jhi + 1);
  it.nkt = jhi < 0 ? 0 : it.ns + max(0, jhi - max(jlo, sinkT) + 1);
  return true;
}

// dQ of query tiles (128 rows) of a query head: items (query tile, query
// head, batch), persistent for dense calls and one CTA per item for packed
// ones, as in the dK/dV kernel.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmDO, BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  chain_allow_next();
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sDO = smem + C::kOffDO;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBarQ);
  uint64_t* qd_full = bars;       // Q and dO landed
  uint64_t* k_full = bars + 1;    // [3] K of a key tile landed
  uint64_t* k_free = bars + 13;   // [3] S and dQ of that tile are done
  uint64_t* v_full = bars + 16;   // [2] V of a key tile landed
  uint64_t* v_free = bars + 18;   // [2] dP of that tile is done
  uint64_t* sa_full = bars + 5;   // S of a key tile is in tensor memory
  uint64_t* st_read = bars + 6;   // S read out (one arrival per compute warp)
  // [2] dP of a key tile is in its buffer / dS written over it (one arrival
  // per compute thread), one barrier per buffer: dP of the next tile is
  // issued before dS of this one is formed, so with one barrier for both
  // buffers a phase could complete twice before a waiter looks
  uint64_t* sb_full = bars + 22;
  uint64_t* p_ready = bars + 20;
  uint64_t* done = bars + 8;      // every product of the item is done
  uint64_t* drain = bars + 9;
  uint64_t* qd_empty = bars + 11; // the item's last products reading Q and dO are done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);
  static_assert(2 * kB + D + kB <= 512, "S, two dP buffers and dQ in tensor memory");
  __shared__ int abort_s;
  volatile int* abort_flag = &abort_s;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int num_items = (p.Sqp / kB) * p.Hq * p.B;

  if (threadIdx.x == 0) {
    mbar_init(qd_full, 1);
    mbar_init(qd_empty, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_free[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_free[s], 1);
      mbar_init(&sb_full[s], 1);
      mbar_init(&p_ready[s], kComputeThreads);
    }
    mbar_init(sa_full, 1);
    mbar_init(st_read, kComputeWarps);
    mbar_init(done, 1);
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
  auto kslot = [&](int u) { return smem + C::kOffKs + (u % 3) * C::kTile; };  // K of key tile u
  auto vslot = [&](int u) { return smem + C::kOffVs + (u & 1) * C::kTile; };  // V of key tile u
  // Tensor memory: S [0,128); dP of key tile u (counted over the CTA's
  // items), then dS over it, in one of two buffers: [128,256) or [384,512);
  // dQ [256,256+D).
  auto dp_col = [&](int u) { return (u & 1) ? 3u * kB : 1u * kB; };

  // Counters over the CTA's items: key tiles (one K and one V load, one set
  // of products each) and items with key tiles (one Q / dO load each).
  if (warp == kWarpProd) {
    // ================================================================ producer
    int qd_loads = 0, issued = 0, k_loads = 0;  // issued: V loads (and key tiles)
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int item = bwd_item_at(n, num_items);
      if (item < 0) break;
      QItem it;
      if (!q_item(p, item, it) || it.nkt == 0) continue;
      // Q and dO are single-buffered: the previous item's last S and dP must
      // be done with them
      if (qd_loads > 0 && !warp_wait(qd_empty, (qd_loads - 1) & 1, abort_flag, p)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx_w(qd_full, 2 * C::kTile);
#pragma unroll
      for (int a = 0; a < C::kAtoms; ++a) {
        tma_load_4d_w(sQ + a * C::kAtomBytes, &tmQ, qd_full, a * 64, it.h,
                      it.sg.q_base + it.q0, it.sg.b_coord);
        tma_load_4d_w(sDO + a * C::kAtomBytes, &tmDO, qd_full, a * 64, it.h,
                      it.sg.q_base + it.q0, it.sg.b_coord);
      }
      ++qd_loads;
      // Warm L2 with the next item's Q and dO (single-buffered, as K and V
      // in the dK/dV kernel).
      {
        QItem nx;
        const int nitem = bwd_item_at(n + 1, num_items);
        if (nitem >= 0 && q_item(p, nitem, nx) && nx.nkt > 0) {
#pragma unroll
          for (int a = 0; a < C::kAtoms; ++a) {
            tma_prefetch_4d_w(&tmQ, a * 64, nx.h, nx.sg.q_base + nx.q0, nx.sg.b_coord);
            tma_prefetch_4d_w(&tmDO, a * 64, nx.h, nx.sg.q_base + nx.q0, nx.sg.b_coord);
          }
        }
      }
      // K of key tile u goes to slot u % 3 once S and dQ of tile u - 3 are
      // done, V to slot u % 2 once dP of tile u - 2 is: both loads run more
      // than a key tile ahead of their first product.
      for (int t = 0; t < it.nkt; ++t) {
        const int u = issued;
        if (u >= 3 && !warp_wait(&k_free[u % 3], ((u / 3) - 1) & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        const int kr = it.sg.k_base + it.tile_at(t) * kB;
        mbar_arrive_expect_tx_w(&k_full[u % 3], C::kTile);
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a)
          tma_load_4d_w(kslot(u) + a * C::kAtomBytes, &tmK, &k_full[u % 3], a * 64, it.hk, kr,
                        it.sg.b_coord);
        ++k_loads;
        if (u >= 2 && !warp_wait(&v_free[u & 1], ((u >> 1) - 1) & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx_w(&v_full[u & 1], C::kTile);
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a)
          tma_load_4d_w(vslot(u) + a * C::kAtomBytes, &tmV, &v_full[u & 1], a * 64, it.hk, kr,
                        it.sg.b_coord);
        ++issued;
      }
    }
    if (qd_loads > 0) warp_wait(qd_full, (qd_loads - 1) & 1, nullptr, p);
    for (int s = 0; s < 3; ++s) {
      const int n_s = (k_loads - s + 2) / 3;
      if (n_s > 0) warp_wait(&k_full[s], (n_s - 1) & 1, nullptr, p);
    }
    for (int s = 0; s < 2; ++s) {
      const int n_s = (issued - s + 1) / 2;
      if (n_s > 0) warp_wait(&v_full[s], (n_s - 1) & 1, nullptr, p);
    }
  } else if (warp == kWarpIssue) {
    // ================================================================ MMA issuer
    // Per key tile t the pipe runs S(t+1), dP(t+1), dQ(t): S of the next
    // tile overwrites S(t) as soon as the compute warps have read it out,
    // and dP(t+1) goes to the other dP buffer, so neither waits for dS(t);
    // dP(t+2) overwrites dS(t) after dQ(t) has read it.  An item's first dQ
    // overwrites the accumulator: it waits for the dS arrival the compute
    // warps make after reading the previous item's dQ out.
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, kB, false);
    constexpr uint32_t idesc_g = idesc_bf16_f32(128, D, true);
    const uint64_t dq = sdesc_sw128(smem_addr(sQ), 16, 1024);
    const uint64_t ddo = sdesc_sw128(smem_addr(sDO), 16, 1024);
    const uint32_t tDQ = tmem + 2 * kB;
    int U = 0;    // key tiles of earlier items
    int qdi = 0;  // items with key tiles before this one
    auto issue_s = [&](int u) -> bool {  // S(u) = Q K(u)^T, over S(u-1) once read out
      if (u > 0 && !warp_wait(st_read, (u - 1) & 1, abort_flag, p)) return false;
      if (!warp_wait(&k_full[u % 3], (u / 3) & 1, abort_flag, p)) return false;
      tc_fence_after_sync();
      const uint64_t dkk = sdesc_sw128(smem_addr(kslot(u)), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t ko = kmajor_step<C::kAtomBytes>(kk);
        mma_bf16_ss_w(tmem, dq + ko, dkk + ko, idesc_s, kk > 0 ? 1u : 0u);
      }
      mma_commit_w(sa_full);
      return true;
    };
    auto issue_dp = [&](int u) -> bool {  // dP(u) = dO V(u)^T (M = queries, N = keys, K = d)
      if (!warp_wait(&v_full[u & 1], (u >> 1) & 1, abort_flag, p)) return false;
      tc_fence_after_sync();
      const uint64_t dvk = sdesc_sw128(smem_addr(vslot(u)), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t ko = kmajor_step<C::kAtomBytes>(kk);
        mma_bf16_ss_w(tmem + dp_col(u), ddo + ko, dvk + ko, idesc_s, kk > 0 ? 1u : 0u);
      }
      mma_commit_w(&sb_full[u & 1]);
      mma_commit_w(&v_free[u & 1]);
      return true;
    };
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int item = bwd_item_at(n, num_items);
      if (item < 0) break;
      QItem it;
      if (!q_item(p, item, it) || it.nkt == 0) continue;
      const int nt = it.nkt;
      ok = warp_wait(qd_full, qdi & 1, abort_flag, p);
      if (ok) tc_fence_after_sync();
      if (ok) ok = issue_s(U) && issue_dp(U);
      for (int t = 0; ok && t < nt; ++t) {
        const int u = U + t;
        // the item's last products reading Q and dO (its last S and dP, issued
        // before): the producer may load the next item's Q and dO
        if (t + 1 == nt) mma_commit_w(qd_empty);
        if (t + 1 < nt && !(issue_s(u + 1) && issue_dp(u + 1))) {
          ok = false;
          break;
        }
        if (!warp_wait(&p_ready[u & 1], (u >> 1) & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        // dQ += dS K(t) (A = dS from tensor memory, K = keys; B = K(t) read along d)
        const uint64_t dkm = sdesc_sw128(smem_addr(kslot(u)), C::kAtomBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kB / 16; ++kk)
          mma_bf16_ts_w(tDQ, tmem + dp_col(u) + packed_col(kk), dkm + kk * (2048 >> 4), idesc_g,
                        (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit_w(&k_free[u % 3]);
      }
      if (ok) mma_commit_w(done);
      U += nt;
      ++qdi;
    }
    mma_commit_w(drain);
    warp_wait(drain, 0, nullptr, p);
  } else if (warp < kComputeWarps) {
    // ================================================================ compute warps
    const int wq = warp & 3, wh = warp >> 2;  // lane quarter, column half
    const int r = wq * 32 + lane;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint64_t sc2 = pf2(p.scale2, p.scale2);
    int U = 0;    // key tiles of earlier items
    int qdi = 0;  // items with key tiles before this one
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int item = bwd_item_at(n, num_items);
      if (item < 0) break;
      QItem it;
      if (!q_item(p, item, it)) continue;
      const int nt = it.nkt;
      const int off = it.sg.Lk - it.sg.Lq;
      const int q_idx = it.q0 + r;
      const size_t vrow = (static_cast<size_t>(it.b) * p.Hq + it.h) * p.Sqp + q_idx;
      const float nlse2 = p.lse2[vrow];  // -LSE2; -inf past Sq: every P of the row is 0
      const float ndval = p.dvec[vrow];  // -D
      const uint64_t nl2 = pf2(nlse2, nlse2), nd2 = pf2(ndval, ndval);
      for (int t = 0; t < nt; ++t) {
        const int u = U + t;
        // P of this warp's 64 columns from S(t), while dQ(t-1) and S(t+1) run
        if (!warp_wait(sa_full, u & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        // column c (key j*128 + c) is visible to this row iff c <= cmax (the
        // key tail, causal) and, with a window, c > cmin or the key is a sink
        const int j = it.tile_at(t);
        int cmax = it.sg.Lk - 1 - j * kB;
        if (p.causal) cmax = min(cmax, q_idx + off - j * kB);
        const int cmin = p.window > 0 ? q_idx + off - p.window - j * kB : -(1 << 30);
        const int csink = p.n_sink - j * kB;  // columns below are sink keys
        uint64_t pp[32];  // P in fp32 pairs
        {
          uint32_t ra[64];
          tmem_ld_x32(taddr + 64 * wh, ra);
          tmem_ld_x32(taddr + 64 * wh + 32, ra + 32);
          tmem_ld_wait_b();
          // S(t) is in registers: S(t+1) may replace it
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(st_read);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            reg_fence_b(ra[2 * e]);
            reg_fence_b(ra[2 * e + 1]);
            float x0, x1;
            pf2_split(pf2_fma(pf2(__uint_as_float(ra[2 * e]), __uint_as_float(ra[2 * e + 1])),
                              sc2, nl2),
                      x0, x1);
            pp[e] = pf2(ex2_approx(x0), ex2_approx(x1));
          }
        }
        // dS = P (dP - D) once dP(t) is in tensor memory
        if (!warp_wait(&sb_full[u & 1], (u >> 1) & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        {
          uint32_t rb[64];
          tmem_ld_x32(taddr + dp_col(u) + 64 * wh, rb);
          tmem_ld_x32(taddr + dp_col(u) + 64 * wh + 32, rb + 32);
          tmem_ld_wait_b();
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int c4 = 2 * wh + jj;
            float pf[32];
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              reg_fence_b(rb[32 * jj + 2 * e]);
              reg_fence_b(rb[32 * jj + 2 * e + 1]);
              const uint64_t g2 = pf2_add(pf2(__uint_as_float(rb[32 * jj + 2 * e]),
                                              __uint_as_float(rb[32 * jj + 2 * e + 1])),
                                          nd2);
              pf2_split(pf2_mul(pp[16 * jj + e], g2), pf[2 * e], pf[2 * e + 1]);
            }
            if (cmax < 32 * c4 + 31 || (cmin >= 32 * c4 && csink < 32 * c4 + 32)) {
              // a chunk the diagonal, the key tail or the window's edge crosses
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const int c = 32 * c4 + e;
                if (c > cmax || (c <= cmin && c >= csink)) pf[e] = 0.f;
              }
            }
            pack32(pf, pk);
            tmem_st_x16(taddr + dp_col(u) + 64 * wh + 16 * jj, pk);
          }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&p_ready[u & 1]);
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (nt > 0) {
        if (!warp_wait(done, qdi & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
      }
      const bool valid = q_idx < it.sg.Lq;
      __nv_bfloat16* dst =
          p.dq + ((static_cast<size_t>(it.sg.q_row0) + q_idx) * p.Hq + it.h) * D;
      constexpr int kHalfChunks = D / 64;
#pragma unroll 1
      for (int c = wh * kHalfChunks; c < (wh + 1) * kHalfChunks; ++c) {
        uint32_t ra[32];
        if (nt > 0) {
          tmem_ld_x32(taddr + 2 * kB + 32 * c, ra);
          tmem_ld_wait_b();
        }
        float f[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          reg_fence_b(ra[e]);
          f[e] = nt > 0 ? __uint_as_float(ra[e]) * p.scale : 0.f;
        }
        uint32_t pk[16];
        pack32(f, pk);
        if (valid) store_row32(dst + 32 * c, pk, p.v8);
      }
      // The next item's first dQ waits for this warp's next arrival, made
      // after the reads of the accumulator above.
      tc_fence_before_sync();
      U += nt;
      if (nt > 0) ++qdi;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 512);
  chain_join_prev();
}

// The dK/dV and dQ kernels of head dimension 64 or 128.
template <int D>
cudaError_t launch_bwd_grads(const BwdParams& p, const BwdLaunch& a, cudaStream_t stream) {
  using C = BwdCfg<D>;
  cudaError_t e;
  // Dense calls: persistent grids (one CTA per SM; every item is about the
  // same work, or ordered longest first under a causal mask).  Packed calls:
  // one CTA per item, so that the hardware hands the next item to whichever
  // SM frees first (item costs follow the sequence lengths).
  const bool packed = a.cu_q != nullptr;
  auto grid_of = [&](long long items) {
    return static_cast<unsigned>(packed ? items
                                        : std::min<long long>(items, std::max(a.num_sms, 1)));
  };
  if (a.Skv > 0) {
    const long long n1 = static_cast<long long>((a.Skv + kB - 1) / kB) * a.Hkv * a.B;
    attn_bwd_dkdv_kernel<D><<<grid_of(n1), kBwdThreads, C::kLaunchKV, stream>>>(
        a.tmQ, a.tmK, a.tmV, a.tmDO, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // dQ as the programmatic dependent of dK/dV (never of the row statistics,
  // which it reads): its CTAs take the SMs that dK/dV CTAs leave.
  const long long n2 = static_cast<long long>(p.Sqp / kB) * a.Hq * a.B;
  if (a.Skv > 0)
    return launch_chained(attn_bwd_dq_kernel<D>, grid_of(n2), C::kLaunchQ, stream, a.tmQ, a.tmK,
                          a.tmV, a.tmDO, p);
  attn_bwd_dq_kernel<D><<<grid_of(n2), kBwdThreads, C::kLaunchQ, stream>>>(a.tmQ, a.tmK, a.tmV,
                                                                          a.tmDO, p);
  return cudaGetLastError();
}


template <int D>
cudaError_t set_bwd_attributes() {
  using C = BwdCfg<D>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kLaunchKV);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(attn_bwd_dq_kernel<D>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, C::kLaunchQ);
  });
  return attr_err;
}

// Row statistics, then the gradient kernels of head dimension D (d = 256:
// attn_bwd256_sm103.cu), then the logit sink's gradient.
template <int D>
cudaError_t launch_bwd_d(const BwdLaunch& a, cudaStream_t stream) {
  if constexpr (D != 256) {
    const cudaError_t attr_err = set_bwd_attributes<D>();
    if (attr_err != cudaSuccess) return attr_err;
  }
  BwdParams p;
  p.dout = static_cast<const __nv_bfloat16*>(a.dout);
  p.o = static_cast<const __nv_bfloat16*>(a.o);
  p.v = static_cast<const __nv_bfloat16*>(a.v);
  p.lse = a.lse;
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.total_q = a.total_q;
  p.total_k = a.total_k;
  p.window = a.window;
  p.n_sink = a.n_sink;
  p.lse2 = a.ws_lse2;
  p.dvec = a.ws_d;
  p.dq = static_cast<__nv_bfloat16*>(a.dq);
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.v8 = (reinterpret_cast<uintptr_t>(a.dq) | reinterpret_cast<uintptr_t>(a.dk) |
          reinterpret_cast<uintptr_t>(a.dv)) % 32 == 0;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Skv = a.Skv;
  p.Sqp = (a.Sq + kB - 1) / kB * kB;
  p.d = D;
  p.scale = a.scale;
  p.scale2 = a.scale * kLog2eB;
  p.causal = a.causal;
  p.wait_limit_ns = kWaitLimitNs;
  p.status = a.status;
  attn_bwd_rowstat_kernel<D><<<1216, 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if constexpr (D == 256) {
    if ((e = launch_bwd256(p, a, stream)) != cudaSuccess) return e;
  } else {
    if ((e = launch_bwd_grads<D>(p, a, stream)) != cudaSuccess) return e;
  }
  if (a.sink != nullptr) {
    attn_bwd_dsink_kernel<<<a.Hq, kSinkThreads, 0, stream>>>(p.lse2, p.dvec, a.sink, a.dsink, a.B,
                                                             a.Hq, p.Sqp);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

size_t bwd_workspace_bytes(int B, int Hq, int Sq) {
  const size_t sqp = (static_cast<size_t>(Sq) + kB - 1) / kB * kB;
  return 2 * static_cast<size_t>(B) * Hq * sqp * sizeof(float);
}

cudaError_t launch_attn_bwd(const BwdLaunch& a, cudaStream_t stream) {
  if (a.d == 128) return launch_bwd_d<128>(a, stream);
  if (a.d == 64) return launch_bwd_d<64>(a, stream);
  if (a.d == 256) return launch_bwd_d<256>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
