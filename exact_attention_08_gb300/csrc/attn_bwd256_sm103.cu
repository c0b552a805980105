// Backward pass at head dimension 256 on sm_103a: dQ, dK and dV of the dense
// exact-attention forward with the masks, packed sequences and fixed
// reduction order of the d = 64 / 128 kernels in attn_bwd_sm103.cu (which
// state the chain rule they follow; "TileLang tutorial, ch.15 Operators:
// Attention", section 5.4 is why no gradient is accumulated atomically).
//
// At d = 256 a 128-row bf16 tile is 64 KB and an fp32 accumulator takes 256
// tensor-memory columns, so the d = 128 layout does not fit:
//   - dK and dV together would fill all 512 columns before any score tile:
//     they come from two launches over the same key tiles (dV, then dK),
//     each recomputing the scores;
//   - four 64 KB tiles exceed the 227 KB of shared memory: the streamed
//     operand comes in 64-row tiles (32 KB) and the A operand of the second
//     product (dO rows for dQ, V rows for dK) is held in tensor memory.
//
// One kernel in three modes, the same products in each:
//   mode  resident R1 (smem)  R2 (tmem)  streamed X (3 slots)  Y (2 slots)  accumulator
//   dQ    Q, 128 rows         dO         K, 64 keys            V            dQ += dS K
//   dK    K, 128 keys         V          Q, 64 queries         dO           dK += dS^T Q
//   dV    K, 128 keys         -          Q, 64 queries         dO           dV += P^T dO
// Per streamed tile t:
//   S  = R1 X(t)^T     M=128, N=64, K=256, both operands K-major in shared memory
//   dP = R2 Y(t)^T     A from tensor memory (dQ and dK only)
//   P  = exp2(S scale log2(e) - LSE log2(e)) under the mask, dS = P (dP - D)
//   ACC += A B         A = dS (dV: P) as bf16 pairs in tensor memory, B = X(t)
//                      (dV: Y(t)) read along d (MN-major), N=256, K=64
// Tensor memory: R2 [0,128) (bf16 pairs), S [128,192), dP and the packed
// operand [192,256), the accumulator [256,512).  S is single: the next S is
// issued as soon as the compute warps have read this one out.
//
// Warps 0-7 compute (warp w: lanes 32 (w % 4) .. +31, columns 32 (w / 4) ..
// +31 of each 64-column tile, 128 (w / 4) .. +127 of the accumulator), 8 TMA
// producer, 9 MMA issuer.  One CTA per item (a 128-row tile of one head).
#include "attn_bwd_common.cuh"

#include <algorithm>
#include <mutex>

namespace attn {
namespace {

constexpr int kD = 256;
constexpr int kT = 64;  // rows of a streamed tile
constexpr int kXSlots = 3;
constexpr int kYSlots = 2;
constexpr int kResAtom = kB * 128;  // one 64-column atom of a 128-row tile (16 KB)
constexpr int kStrAtom = kT * 128;  // one atom of a 64-row tile (8 KB)
constexpr int kResBytes = kB * kD * 2;
constexpr int kStrBytes = kT * kD * 2;
constexpr int kVec = kT * 4;  // one fp32 vector of a streamed tile
constexpr int kOffR1 = 0;
constexpr int kOffX = kOffR1 + kResBytes;
constexpr int kOffY = kOffX + kXSlots * kStrBytes;
constexpr int kOffVec = kOffY + kYSlots * kStrBytes;  // per X slot: -LSE2, -D
constexpr int kOffBar = kOffVec + kXSlots * 2 * kVec;
constexpr int kNumBars = 20;
constexpr int kSmem256 = kOffBar + kNumBars * 8;
static_assert(kSmem256 <= 227 * 1024, "shared memory");
static_assert(kOffX % 1024 == 0 && kOffY % 1024 == 0, "swizzle atoms");

constexpr uint32_t kColR2 = 0, kColS = 128, kColP = 192, kColAcc = 256;

enum : int { kModeDQ = 0, kModeDK = 1, kModeDV = 2 };

// K-step kk (16 columns) of a 64-column tile written as bf16 pairs in place
// of its fp32 values: each column half (32 values) packs into the first 16
// columns of that half, so the warp that reads a half is the one that writes it.
__device__ __forceinline__ uint32_t packed64(int kk) {
  return static_cast<uint32_t>(32 * (kk / 2) + 8 * (kk % 2));
}

// One item: the resident 128-row tile and the streamed tiles it meets.
struct Work256 {
  int b, h, hk;  // sequence, query head (dQ), key head
  int r0;        // first row of the resident tile in its sequence
  int nt;        // streamed tiles
  int lo, ns;    // dQ: first window tile past the sink tiles, sink tiles; dK/dV: first query tile
  int nq;        // dK/dV: query tiles per query head
  SeqGeo sg;
  // first row (in its sequence) and head of streamed tile n
  __device__ __forceinline__ void tile(int n, int G, int dq_mode, int& row, int& head) const {
    if (dq_mode) {
      row = (n < ns ? n : lo + (n - ns)) * kT;
      head = hk;
    } else {
      row = (lo + n % nq) * kT;
      head = hk * G + n / nq;
    }
  }
};

// Item order as in the d = 128 kernels: under a causal mask the longest
// items first, otherwise the tiles of one (sequence, head) adjacent.  False
// for a tile past its sequence (nothing to write).
template <int kMode>
__device__ __forceinline__ bool work256(const BwdParams& p, int item, Work256& w) {
  if (kMode == kModeDQ) {
    const int nqt_all = p.Sqp / kB;
    int qt;
    if (p.causal) {
      qt = nqt_all - 1 - item / (p.B * p.Hq);
      w.h = (item / p.B) % p.Hq;
      w.b = item % p.B;
    } else {
      qt = item % nqt_all;
      w.h = (item / nqt_all) % p.Hq;
      w.b = item / (nqt_all * p.Hq);
    }
    w.hk = w.h / (p.Hq / p.Hkv);
    w.r0 = qt * kB;
    if (!seq_geo(p, w.b, w.sg, false) || w.r0 >= w.sg.Lq) return false;
    const int off = w.sg.Lk - w.sg.Lq;
    // the key tiles the rows see: the sink tiles, then from the first key
    // above the first row's window bound to the last key any row sees
    int jhi = -1;
    if (w.sg.Lk > 0) {
      int kmax = w.sg.Lk - 1;
      if (p.causal) kmax = min(kmax, min(w.r0 + kB - 1, w.sg.Lq - 1) + off);
      jhi = kmax >= 0 ? kmax / kT : -1;
    }
    int jlo = 0, sinkT = 0;
    if (p.window > 0) {
      const int lo = w.r0 + off - p.window;  // keys above lo are in the first row's window
      jlo = lo < 0 ? 0 : (lo + 1) / kT;
      sinkT = (p.n_sink + kT - 1) / kT;
    }
    w.ns = min(sinkT, jhi + 1);
    w.lo = max(jlo, sinkT);
    w.nt = jhi < 0 ? 0 : w.ns + max(0, jhi - w.lo + 1);
    w.nq = 0;
  } else {
    const int nkt_all = (p.Skv + kB - 1) / kB;
    int kt;
    if (p.causal) {
      kt = item / (p.B * p.Hkv);
      w.hk = (item / p.B) % p.Hkv;
      w.b = item % p.B;
    } else {
      kt = item % nkt_all;
      w.hk = (item / nkt_all) % p.Hkv;
      w.b = item / (nkt_all * p.Hkv);
    }
    w.h = -1;
    w.r0 = kt * kB;
    if (!seq_geo(p, w.b, w.sg, false) || w.r0 >= w.sg.Lk) return false;
    const int off = w.sg.Lk - w.sg.Lq;
    // the query tiles that see a key of the tile: from the first query that
    // sees key r0 (causal) to the last that sees key r0 + 127 (window; a
    // tile holding sink keys is seen to the end)
    int qt_lo = 0, qt_hi = (w.sg.Lq + kT - 1) / kT - 1;
    if (p.causal) {
      const int qmin = w.r0 - off;
      qt_lo = qmin <= 0 ? 0 : qmin / kT;
    }
    if (p.window > 0 && w.r0 >= p.n_sink) {
      const int qmax = w.r0 + kB - 1 - off + p.window - 1;
      qt_hi = qmax < 0 ? -1 : min(qt_hi, qmax / kT);
    }
    w.lo = qt_lo;
    w.nq = qt_hi >= qt_lo ? qt_hi - qt_lo + 1 : 0;
    w.nt = (p.Hq / p.Hkv) * w.nq;  // (query head, query tile) pairs, head-major
    w.ns = 0;
  }
  return true;
}

template <int kMode>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd256_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmDO, BwdParams p) {
  constexpr bool kDQ = kMode == kModeDQ;
  constexpr bool kHasDP = kMode != kModeDV;
  extern __shared__ uint8_t smem[];
  chain_allow_next();
  // The layout fills shared memory with no room to round the window up to
  // the swizzle atom: a window off the boundary is reported, not used.
  if (smem_addr(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    chain_join_prev();
    return;
  }
  Work256 w;
  if (!work256<kMode>(p, static_cast<int>(blockIdx.x), w)) {
    chain_join_prev();
    return;
  }
  const int G = p.Hq / p.Hkv;
  const int nt = w.nt;
  uint8_t* sR1 = smem + kOffR1;
  auto sX = [&](int s) { return smem + kOffX + s * kStrBytes; };
  auto sY = [&](int s) { return smem + kOffY + s * kStrBytes; };
  auto sVec = [&](int s) { return smem + kOffVec + s * 2 * kVec; };
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* r1_full = bars;       // resident tile landed
  uint64_t* r2_ready = bars + 1;  // R2 in tensor memory (one arrival per compute thread)
  uint64_t* x_full = bars + 2;    // [3]
  uint64_t* x_empty = bars + 5;   // [3]
  uint64_t* y_full = bars + 8;    // [2]
  uint64_t* y_empty = bars + 10;  // [2]
  uint64_t* sa_full = bars + 12;  // S in tensor memory
  uint64_t* st_read = bars + 13;  // S read out (one arrival per compute warp)
  uint64_t* sb_full = bars + 14;  // dP in tensor memory (dV: its columns free)
  uint64_t* pb_ready = bars + 15; // packed operand written (one arrival per compute thread)
  uint64_t* done = bars + 16;     // every product done
  uint64_t* drain = bars + 17;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 18);
  int* abort_s = reinterpret_cast<int*>(bars + 19);
  volatile int* abort_flag = abort_s;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(r1_full, 1);
    mbar_init(r2_ready, kComputeThreads);
    for (int s = 0; s < kXSlots; ++s) {
      mbar_init(&x_full[s], 1);
      mbar_init(&x_empty[s], 1);
    }
    for (int s = 0; s < kYSlots; ++s) {
      mbar_init(&y_full[s], 1);
      mbar_init(&y_empty[s], 1);
    }
    mbar_init(sa_full, 1);
    mbar_init(st_read, kComputeWarps);
    mbar_init(sb_full, 1);
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

  if (warp == kWarpProd) {
    // ================================================================ producer
    int nx = 0, ny = 0;  // loads issued into the X and Y rings
    if (nt > 0) {
      const CUtensorMap* m1 = kDQ ? &tmQ : &tmK;
      const CUtensorMap* mx = kDQ ? &tmK : &tmQ;
      const CUtensorMap* my = kDQ ? &tmV : &tmDO;
      const int base1 = kDQ ? w.sg.q_base : w.sg.k_base;
      const int basex = kDQ ? w.sg.k_base : w.sg.q_base;
      mbar_arrive_expect_tx_w(r1_full, kResBytes);
#pragma unroll
      for (int a = 0; a < kD / 64; ++a)
#pragma unroll
        for (int hf = 0; hf < kB / kT; ++hf)
          tma_load_4d_w(sR1 + a * kResAtom + hf * kStrAtom, m1, r1_full, a * 64,
                        kDQ ? w.h : w.hk, base1 + w.r0 + hf * kT, w.sg.b_coord);
      for (int n = 0; n < nt; ++n) {
        int row, head;
        w.tile(n, G, kDQ, row, head);
        const int xs = n % kXSlots;
        if (n >= kXSlots && !warp_wait(&x_empty[xs], ((n / kXSlots) - 1) & 1, abort_flag, p))
          break;
        mbar_arrive_expect_tx_w(&x_full[xs], kStrBytes + (kDQ ? 0 : 2 * kVec));
#pragma unroll
        for (int a = 0; a < kD / 64; ++a)
          tma_load_4d_w(sX(xs) + a * kStrAtom, mx, &x_full[xs], a * 64, head, basex + row,
                        w.sg.b_coord);
        if (!kDQ) {
          const size_t vrow = (static_cast<size_t>(w.b) * p.Hq + head) * p.Sqp + row;
          bulk_load_1d_w(sVec(xs), p.lse2 + vrow, kVec, &x_full[xs]);
          bulk_load_1d_w(sVec(xs) + kVec, p.dvec + vrow, kVec, &x_full[xs]);
        }
        ++nx;
        const int ys = n % kYSlots;
        if (n >= kYSlots && !warp_wait(&y_empty[ys], ((n / kYSlots) - 1) & 1, abort_flag, p))
          break;
        mbar_arrive_expect_tx_w(&y_full[ys], kStrBytes);
#pragma unroll
        for (int a = 0; a < kD / 64; ++a)
          tma_load_4d_w(sY(ys) + a * kStrAtom, my, &y_full[ys], a * 64, head, basex + row,
                        w.sg.b_coord);
        ++ny;
      }
      // Let every copy issued land before the CTA can leave.
      warp_wait(r1_full, 0, nullptr, p);
      for (int s = 0; s < kXSlots; ++s) {
        const int c = (nx - s + kXSlots - 1) / kXSlots;  // loads into slot s
        if (c > 0) warp_wait(&x_full[s], (c - 1) & 1, nullptr, p);
      }
      for (int s = 0; s < kYSlots; ++s) {
        const int c = (ny - s + kYSlots - 1) / kYSlots;
        if (c > 0) warp_wait(&y_full[s], (c - 1) & 1, nullptr, p);
      }
    }
  } else if (warp == kWarpIssue) {
    // ================================================================ MMA issuer
    // Per streamed tile t: S(t+1) once S(t) is read out, ACC(t) once its
    // operand is packed, dP(t+1) over the packed operand ACC(t) has read.
    if (nt > 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kT, false);
      constexpr uint32_t idesc_a = idesc_bf16_f32(128, kD, true);
      const uint64_t d1 = sdesc_sw128(smem_addr(sR1), 16, 1024);
      const uint32_t tR2 = tmem + kColR2, tS = tmem + kColS, tP = tmem + kColP,
                     tAcc = tmem + kColAcc;
      auto issue_s = [&](int n) -> bool {  // S(n) = R1 X(n)^T
        const int xs = n % kXSlots;
        if (!warp_wait(&x_full[xs], (n / kXSlots) & 1, abort_flag, p)) return false;
        tc_fence_after_sync();
        const uint64_t dx = sdesc_sw128(smem_addr(sX(xs)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_bf16_ss_w(tS, d1 + kmajor_step<kResAtom>(kk), dx + kmajor_step<kStrAtom>(kk),
                        idesc_s, kk > 0 ? 1u : 0u);
        mma_commit_w(sa_full);
        return true;
      };
      auto issue_dp = [&](int n) -> bool {  // dP(n) = R2 Y(n)^T; dV: the packed columns free
        if (!kHasDP) {
          mma_commit_w(sb_full);
          return true;
        }
        const int ys = n % kYSlots;
        if (!warp_wait(&y_full[ys], (n / kYSlots) & 1, abort_flag, p)) return false;
        tc_fence_after_sync();
        const uint64_t dy = sdesc_sw128(smem_addr(sY(ys)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_bf16_ts_w(tP, tR2 + 8 * kk, dy + kmajor_step<kStrAtom>(kk), idesc_s,
                        kk > 0 ? 1u : 0u);
        mma_commit_w(sb_full);
        mma_commit_w(&y_empty[ys]);
        return true;
      };
      bool ok = warp_wait(r1_full, 0, abort_flag, p);
      if (ok && kHasDP) ok = warp_wait(r2_ready, 0, abort_flag, p);
      if (ok) tc_fence_after_sync();
      ok = ok && issue_s(0) && issue_dp(0);
      for (int n = 0; ok && n < nt; ++n) {
        if (n + 1 < nt) {
          if (!warp_wait(st_read, n & 1, abort_flag, p) || !issue_s(n + 1)) {
            ok = false;
            break;
          }
        }
        if (!kHasDP && !warp_wait(&y_full[n % kYSlots], (n / kYSlots) & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        if (!warp_wait(pb_ready, n & 1, abort_flag, p)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint8_t* bsrc = kHasDP ? sX(n % kXSlots) : sY(n % kYSlots);
        const uint64_t db = sdesc_sw128(smem_addr(bsrc), kStrAtom, 1024);
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          mma_bf16_ts_w(tAcc, tP + packed64(kk), db + kk * (2048 >> 4), idesc_a,
                        (n > 0 || kk > 0) ? 1u : 0u);
        // the X slot's last reader (its vectors were read before the packed
        // operand was published); dV: the Y slot's too
        mma_commit_w(&x_empty[n % kXSlots]);
        if (!kHasDP) mma_commit_w(&y_empty[n % kYSlots]);
        if (n + 1 < nt && !issue_dp(n + 1)) {
          ok = false;
          break;
        }
      }
      if (ok) mma_commit_w(done);
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
    const int off = w.sg.Lk - w.sg.Lq;
    const int ridx = w.r0 + r;  // this thread's query (dQ) or key (dK, dV) in its sequence
    const bool rvalid = kDQ ? ridx < w.sg.Lq : ridx < w.sg.Lk;
    bool ok = true;
    // R2 (dO rows for dQ, V rows for dK) into tensor memory as bf16 pairs:
    // this warp's 128 of the row's 256 elements, zeros past the sequence
    if (kHasDP && nt > 0) {
      const __nv_bfloat16* src =
          kDQ ? p.dout + ((static_cast<size_t>(w.sg.q_row0) + ridx) * p.Hq + w.h) * kD
              : p.v + ((static_cast<size_t>(w.sg.k_row0) + ridx) * p.Hkv + w.hk) * kD;
      const uint4* s4 = reinterpret_cast<const uint4*>(src + 128 * wh);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t v32[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 x = rvalid ? s4[8 * hf + i] : make_uint4(0u, 0u, 0u, 0u);
          v32[4 * i] = x.x;
          v32[4 * i + 1] = x.y;
          v32[4 * i + 2] = x.z;
          v32[4 * i + 3] = x.w;
        }
        tmem_st_x32(taddr + kColR2 + 64 * wh + 32 * hf, v32);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(r2_ready);
    }
    // dQ: the row's -LSE2 and -D (-inf past the queries: every P of the row is 0)
    uint64_t nl_row = 0, nd_row = 0;
    if (kDQ) {
      const size_t vrow = (static_cast<size_t>(w.b) * p.Hq + w.h) * p.Sqp + ridx;
      nl_row = pf2(p.lse2[vrow], p.lse2[vrow]);
      nd_row = pf2(p.dvec[vrow], p.dvec[vrow]);
    }
    const int c0 = 32 * wh;  // this warp's first column of a streamed tile
    for (int n = 0; n < nt; ++n) {
      int row, head;
      w.tile(n, G, kDQ, row, head);
      if (!warp_wait(sa_full, n & 1, abort_flag, p) ||
          (!kDQ && !warp_wait(&x_full[n % kXSlots], (n / kXSlots) & 1, abort_flag, p))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t ra[32];
      uint64_t nl[16];
      tmem_ld_x32(taddr + kColS + c0, ra);
      if (!kDQ) lds_chunk(smem_addr(sVec(n % kXSlots)) + 4 * c0, nl);
      tmem_ld_wait_x32(ra);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(st_read);
      float pf[32];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float x0, x1;
        pf2_split(pf2_fma(pf2(__uint_as_float(ra[2 * e]), __uint_as_float(ra[2 * e + 1])), sc2,
                          kDQ ? nl_row : nl[e]),
                  x0, x1);
        pf[2 * e] = ex2_approx(x0);
        pf[2 * e + 1] = ex2_approx(x1);
      }
      // the mask: column c of the tile is row + c of the streamed side
      if (kDQ) {
        // keys: visible iff c <= cmax (key tail, causal) and, with a window,
        // c > cmin or the key is a sink
        int cmax = w.sg.Lk - 1 - row;
        if (p.causal) cmax = min(cmax, ridx + off - row);
        const int cmin = p.window > 0 ? ridx + off - p.window - row : -(1 << 30);
        const int csink = p.n_sink - row;
        if (cmax < c0 + 31 || (cmin >= c0 && csink < c0 + 32)) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int c = c0 + e;
            if (c > cmax || (c <= cmin && c >= csink)) pf[e] = 0.f;
          }
        }
      } else {
        // queries: visible iff cmin <= c (causal) and c <= cmax (the window,
        // not for sink keys); keys past the sequence see nothing
        int cmin = p.causal ? ridx - off - row : -(1 << 30);
        const int cmax = (p.window > 0 && ridx >= p.n_sink) ? ridx - off + p.window - 1 - row
                                                             : (1 << 30);
        if (!rvalid) cmin = 1 << 30;
        if (cmin > c0 || cmax < c0 + 31) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int c = c0 + e;
            if (c < cmin || c > cmax) pf[e] = 0.f;
          }
        }
      }
      if (!warp_wait(sb_full, n & 1, abort_flag, p)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t pk[16];
      if (!kHasDP) {
        pack32(pf, pk);
      } else {
        uint32_t rb[32];
        uint64_t nd[16];
        tmem_ld_x32(taddr + kColP + c0, rb);
        if (!kDQ) lds_chunk(smem_addr(sVec(n % kXSlots)) + kVec + 4 * c0, nd);
        tmem_ld_wait_x32(rb);
        float g[32];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint64_t g2 = pf2_add(pf2(__uint_as_float(rb[2 * e]), __uint_as_float(rb[2 * e + 1])),
                                      kDQ ? nd_row : nd[e]);
          pf2_split(pf2_mul(pf2(pf[2 * e], pf[2 * e + 1]), g2), g[2 * e], g[2 * e + 1]);
        }
        pack32(g, pk);
      }
      tmem_st_x16(taddr + kColP + c0, pk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(pb_ready);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && nt > 0) {
      ok = warp_wait(done, 0, abort_flag, p);
      tc_fence_after_sync();
    }
    if (ok) {
      __nv_bfloat16* dst =
          kDQ ? p.dq + ((static_cast<size_t>(w.sg.q_row0) + ridx) * p.Hq + w.h) * kD
              : (kMode == kModeDK ? p.dk : p.dv) +
                    ((static_cast<size_t>(w.sg.k_row0) + ridx) * p.Hkv + w.hk) * kD;
      const float mul = kMode == kModeDV ? 1.f : p.scale;
#pragma unroll 1
      for (int c = 4 * wh; c < 4 * wh + 4; ++c) {  // 32-column chunks of this warp's half
        uint32_t ra[32];
        if (nt > 0) {
          tmem_ld_x32(taddr + kColAcc + 32 * c, ra);
          tmem_ld_wait_x32(ra);
        }
        float f[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = nt > 0 ? __uint_as_float(ra[e]) * mul : 0.f;
        uint32_t pk[16];
        pack32(f, pk);
        if (rvalid) store_row32(dst + 32 * c, pk, p.v8);
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 512);
  chain_join_prev();
}

// chained: launched as the programmatic dependent of the gradient kernel
// before it (never of the row statistics, which every mode reads).
template <int kMode>
cudaError_t launch_mode(const BwdParams& p, const BwdLaunch& a, long long items, bool chained,
                        cudaStream_t stream) {
  if (chained)
    return launch_chained(attn_bwd256_kernel<kMode>, static_cast<unsigned>(items), kSmem256,
                          stream, a.tmQ, a.tmK, a.tmV, a.tmDO, p);
  attn_bwd256_kernel<kMode><<<static_cast<unsigned>(items), kBwdThreads, kSmem256, stream>>>(
      a.tmQ, a.tmK, a.tmV, a.tmDO, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd256(const BwdParams& p, const BwdLaunch& a, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_bwd256_kernel<kModeDQ>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem256);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(attn_bwd256_kernel<kModeDK>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem256);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(attn_bwd256_kernel<kModeDV>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem256);
  });
  if (attr_err != cudaSuccess) return attr_err;
  cudaError_t e;
  if (a.Skv > 0) {
    const long long n1 = static_cast<long long>((a.Skv + kB - 1) / kB) * a.Hkv * a.B;
    if ((e = launch_mode<kModeDV>(p, a, n1, false, stream)) != cudaSuccess) return e;
    if ((e = launch_mode<kModeDK>(p, a, n1, true, stream)) != cudaSuccess) return e;
  }
  const long long n2 = static_cast<long long>(p.Sqp / kB) * a.Hq * a.B;
  return launch_mode<kModeDQ>(p, a, n2, a.Skv > 0, stream);
}

}  // namespace attn
