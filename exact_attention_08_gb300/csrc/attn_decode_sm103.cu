// One-token decode over a paged KV cache, split-KV (Flash-Decoding) with a
// log-sum-exp merge ("TileLang tutorial, ch.15 Operators: Attention",
// sections 4.6, 4.8(2)-(3) and 5.4; "learn-cuda-from-scratch, ch.12
// FlashAttention", sections 12.9.3-12.9.4).
//
// Split kernel: one CTA per (split, KV head, request, head chunk).  It serves
// the query heads of one KV head (grouped-query attention reads each KV page
// once for the whole group, ch.15 section 4.8(1)).  The keys of request b are
// cut at page granularity: np = ceil(L_b / 16) pages, pps = ceil(np / S) pages
// per split, split s covers pages [s*pps, min((s+1)*pps, np)).
//   warp 0       TMA producer: looks each logical page up in the page table
//                and loads its K and V slices (16 tokens x d of this KV head)
//                through a 4-D tensor map over the page pool into a 6-stage
//                shared-memory ring (no tensor-map rewriting: the physical
//                page index is simply the outermost coordinate);
//   warps 1-2    consumers: warp w takes pages w, w+2, ... of the split and
//                runs its own online softmax over them, with the two small
//                products on mma.sync (queries of the group as the 16-row
//                operand, the page's 16 tokens as the other dimension);
//                then the two warps merge their (m, l, O) states in shared
//                memory and write the split's normalised output and natural
//                log-sum-exp to the workspace.
// Combine kernel: per (request, query head), weights w_s = exp(lse_s - M)
// with M the largest split lse, summed in ascending split order, so the
// result does not depend on which CTA finished first.
//
// The work is bound by HBM bandwidth: every KV byte is read once.  Small CTAs
// (three warps, a 48 KB ring at d = 128) run four to an SM, so that one CTA's
// ramp-up and drain overlap the others' streaming: 192 KB of pages in flight
// per SM (measured against two CTAs of five warps and a 64 KB ring: 0.845
// against 0.745 of the copy bandwidth).  A one-block kernel first orders the
// requests longest first, and the split kernel takes its request from that
// order, so that the short requests' CTAs fill the end of the grid instead
// of a long one running alone there.
#include "attn_internal.h"
#include "sm103_ptx.cuh"

#include <cuda_bf16.h>
#include <mutex>

namespace attn {
namespace {

using namespace ptx;

constexpr int kPage = 16;            // tokens per page
constexpr int kStagesDec = 6;        // page ring depth
constexpr int kConsumers = 2;        // consumer warps
constexpr int kDecCtasPerSm = 4;     // resident split CTAs per SM (registers and ring)
// Consumer warp w takes the pages i = w (mod kConsumers); with the ring depth a
// multiple of that count, every ring slot always goes to the same warp, so a
// warp waits for the phases of a slot in order (a parity wait on a later
// phase would otherwise pass before the earlier one completed).
static_assert(kStagesDec % kConsumers == 0, "a ring slot must always go to the same consumer");
constexpr int kDecThreads = 32 * (1 + kConsumers);
constexpr int kHeadsPerCta = 16;     // query heads served per CTA (mma M)
constexpr float kLog2eDec = 1.4426950408889634f;

template <int D>
struct DecCfg {
  static constexpr int kAtoms = D / 64;
  static constexpr int kBoxBytes = kPage * 128;               // 16 tokens x 64 bf16
  static constexpr int kSliceBytes = kAtoms * kBoxBytes;      // K (or V) slice of one page
  static constexpr int kStageBytes = 2 * kSliceBytes;         // K then V
  static constexpr int kRingBytes = kStagesDec * kStageBytes;
  // merge area reuses the ring: per warp m[16], l[16], O[16][D]
  static constexpr int kMergeBytes = kConsumers * (2 * kHeadsPerCta + kHeadsPerCta * D) * 4;
  static_assert(kMergeBytes <= kRingBytes, "merge area must fit in the ring");
  static constexpr int kOffBar = kRingBytes;
  static constexpr int kSmemBytes = kOffBar + 2 * kStagesDec * 8 + 1024;
};

// Requests longest first: a counting sort of the batch on its page counts
// (descending; when there are more page counts than buckets, buckets of
// equal width), one block.  The split kernel takes its request from this
// order, so the hardware hands out the longest requests' CTAs first and the
// short ones fill the end (the same result whatever the order: every CTA
// computes its own split, and the merge order is fixed).
constexpr int kOrderBuckets = 4096;
constexpr int kOrderThreads = 1024;
__global__ void __launch_bounds__(kOrderThreads)
    attn_decode_order_kernel(const int* __restrict__ seqlens, int B, int max_pages, int* order) {
  __shared__ int cnt[kOrderBuckets];
  __shared__ int wsum[kOrderThreads / 32];
  const int t = threadIdx.x;
  const int nb = min(max_pages + 1, kOrderBuckets);
  for (int i = t; i < kOrderBuckets; i += kOrderThreads) cnt[i] = 0;
  __syncthreads();
  auto bucket = [&](int b) {  // bucket 0: the most pages
    const int L = seqlens[b];
    const int np = L <= 0 ? 0 : min((L + 15) / 16, max_pages);
    const long long k = static_cast<long long>(max_pages - np) * nb / (max_pages + 1);
    return static_cast<int>(k < nb - 1 ? k : nb - 1);
  };
  for (int b = t; b < B; b += kOrderThreads) atomicAdd(&cnt[bucket(b)], 1);
  __syncthreads();
  // Exclusive scan of the counts: four buckets a thread, then across lanes
  // and warps.
  constexpr int kPer = kOrderBuckets / kOrderThreads;
  int local[kPer], run = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    local[j] = run;
    run += cnt[t * kPer + j];
  }
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if ((t & 31) >= o) incl += v;
  }
  if ((t & 31) == 31) wsum[t >> 5] = incl;
  __syncthreads();
  if (t < 32) {
    const int v = wsum[t];
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (t >= o) x += y;
    }
    wsum[t] = x - v;
  }
  __syncthreads();
  const int base = wsum[t >> 5] + (incl - run);
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kPer; ++j) cnt[t * kPer + j] = base + local[j];
  __syncthreads();
  for (int b = t; b < B; b += kOrderThreads) order[atomicAdd(&cnt[bucket(b)], 1)] = b;
}

struct DecParams {
  const __nv_bfloat16* q;
  const int* page_table;
  const int* seqlens;
  float* ws_o;
  float* ws_lse;
  const int* order;  // [B] requests longest first (the grid's z order)
  int B, Hq, Hkv, G, n_hchunks, max_pages, num_pages, num_splits;
  float scale, scale2;
  uint64_t wait_limit_ns;
  int* status;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of (token, element e) inside a 16-token x 64-element box laid
// out by TMA with the 128-byte swizzle (16-byte chunks XOR token % 8).
__device__ __forceinline__ uint32_t swz(int token, int e) {
  return token * 128 + ((((e >> 3) ^ token) & 7) << 4) + (e & 7) * 2;
}

template <int D>
__global__ void __launch_bounds__(kDecThreads, kDecCtasPerSm)
    attn_decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV, const DecParams p) {
  using C = DecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* empty = full + kStagesDec;
  __shared__ int abort_flag_s;
  volatile int* abort_flag = &abort_flag_s;

  const int split = blockIdx.x;
  const int hkv = blockIdx.y / p.n_hchunks;
  const int hchunk = blockIdx.y % p.n_hchunks;
  // Launched as a programmatic dependent of the order kernel: the launch
  // overlaps it, and this waits for its result.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = p.order[blockIdx.z];
  const int g0 = hchunk * kHeadsPerCta;                  // first group member served
  const int nh = min(kHeadsPerCta, p.G - g0);            // query heads served
  const int h0 = hkv * p.G + g0;                         // first query head served

  int L = p.seqlens[b];
  if (L < 0 || L > p.max_pages * kPage) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusBadInput);
    L = max(0, min(L, p.max_pages * kPage));
  }
  const int np = (L + kPage - 1) / kPage;
  const int pps = (np + p.num_splits - 1) / p.num_splits;
  const int pg0 = min(split * pps, np);
  const int pg1 = min(pg0 + pps, np);
  const int npg = pg1 - pg0;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    abort_flag_s = 0;
    for (int s = 0; s < kStagesDec; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ============================================================ producer
    if (lane == 0 && npg > 0) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const int* row = p.page_table + static_cast<size_t>(b) * p.max_pages;
      int page_next = row[pg0];  // each page index read one page ahead of its loads
      for (int i = 0; i < npg; ++i) {
        const int s = i % kStagesDec;
        int page = page_next;
        if (i + 1 < npg) page_next = row[pg0 + i + 1];
        if (!mbar_wait(&empty[s], ((i / kStagesDec) & 1) ^ 1, abort_flag, p.wait_limit_ns)) {
          atomicOr(p.status, kStatusTimeout);
          *abort_flag = 1;
          break;
        }
        if (page < 0 || page >= p.num_pages) {
          atomicOr(p.status, kStatusBadInput);
          page = p.num_pages;  // past the pool: the copy reads zeros
        }
        uint8_t* st = smem + s * C::kStageBytes;
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a) {
          tma_load_4d(st + a * C::kBoxBytes, &tmK, &full[s], a * 64, hkv, 0, page);
          tma_load_4d(st + C::kSliceBytes + a * C::kBoxBytes, &tmV, &full[s], a * 64, hkv, 0, page);
        }
      }
    }
    __syncwarp();
  } else {
    // ============================================================ consumers
    const int cw = warp - 1;
    const int r_lo = lane >> 2;       // mma rows held by this lane: r_lo, r_lo + 8
    const int cpair = (lane & 3) * 2; // mma columns held: cpair, cpair + 1

    // Q fragments (A operand, rows = query heads of the group), loaded once.
    uint32_t qa[D / 16][4];
    {
      const __nv_bfloat16* qb = p.q + (static_cast<size_t>(b) * p.Hq + h0) * D;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int f = 0; f < 4; ++f) {
          const int rr = r_lo + ((f & 1) ? 8 : 0);
          const int cc = kk * 16 + cpair + ((f & 2) ? 8 : 0);
          uint32_t v = 0;
          if (rr < nh) v = *reinterpret_cast<const uint32_t*>(qb + static_cast<size_t>(rr) * D + cc);
          qa[kk][f] = v;
        }
      }
    }

    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
    const float scale2 = p.scale2;

    // ldmatrix addressing: thread t supplies row (t % 8) of matrix (t / 8)
    const int mi = lane >> 3, rr8 = lane & 7;

    for (int i = cw; i < npg; i += kConsumers) {
      const int s = i % kStagesDec;
      bool ok = mbar_wait(&full[s], (i / kStagesDec) & 1, abort_flag, p.wait_limit_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) {
          atomicOr(p.status, kStatusTimeout);
          *abort_flag = 1;
        }
        break;
      }
      const uint32_t kst = smem_addr(smem + s * C::kStageBytes);
      const uint32_t vst = kst + C::kSliceBytes;

      // ---- S[16 heads x 16 tokens] = Q K^T
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int tok = rr8 + ((mi & 2) ? 8 : 0);
        const int e = kk * 16 + ((mi & 1) ? 8 : 0);
        uint32_t b00, b01, b10, b11;
        ldsm_x4(kst + (e / 64) * C::kBoxBytes + swz(tok, e % 64), b00, b01, b10, b11);
        mma16816(sc[0], qa[kk], b00, b01);
        mma16816(sc[1], qa[kk], b10, b11);
      }
      // ---- mask tokens past the request's length
      const int tok_base = (pg0 + i) * kPage;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (tok_base + nt * 8 + cpair + (e & 1) >= L) sc[nt][e] = -INFINITY;

      // ---- online softmax over the page (rows r_lo: e = 0,1; r_lo + 8: e = 2,3)
      float mx_lo = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float mx_hi = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
      const float ms_lo = (mn_lo == -INFINITY) ? 0.f : mn_lo * scale2;
      const float ms_hi = (mn_hi == -INFINITY) ? 0.f : mn_hi * scale2;
      const float a_lo = ex2_approx(fmaf(m_lo, scale2, -ms_lo));
      const float a_hi = ex2_approx(fmaf(m_hi, scale2, -ms_hi));
      m_lo = mn_lo;
      m_hi = mn_hi;
      uint32_t pa[4];
      float ps_lo = 0.f, ps_hi = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float p0 = ex2_approx(fmaf(sc[nt][0], scale2, -ms_lo));
        const float p1 = ex2_approx(fmaf(sc[nt][1], scale2, -ms_lo));
        const float p2 = ex2_approx(fmaf(sc[nt][2], scale2, -ms_hi));
        const float p3 = ex2_approx(fmaf(sc[nt][3], scale2, -ms_hi));
        ps_lo += p0 + p1;
        ps_hi += p2 + p3;
        pa[nt * 2 + 0] = pack_bf16x2(p0, p1);  // rows r_lo, tokens of n-tile nt
        pa[nt * 2 + 1] = pack_bf16x2(p2, p3);  // rows r_lo + 8
      }
      l_lo = l_lo * a_lo + ps_lo;
      l_hi = l_hi * a_hi + ps_hi;
      // A fragment of P: {rows lo, k 0-7}, {rows hi, k 0-7}, {rows lo, k 8-15}, {rows hi, k 8-15}
      const uint32_t afr[4] = {pa[0], pa[1], pa[2], pa[3]};

      // ---- O = alpha O + P V
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= a_lo;
        o[n][1] *= a_lo;
        o[n][2] *= a_hi;
        o[n][3] *= a_hi;
      }
#pragma unroll
      for (int n2 = 0; n2 < D / 16; ++n2) {
        const int tok = rr8 + ((mi & 1) ? 8 : 0);
        const int e = n2 * 16 + ((mi & 2) ? 8 : 0);
        uint32_t b0a, b1a, b0b, b1b;
        ldsm_x4_t(vst + (e / 64) * C::kBoxBytes + swz(tok, e % 64), b0a, b1a, b0b, b1b);
        mma16816(o[2 * n2], afr, b0a, b1a);
        mma16816(o[2 * n2 + 1], afr, b0b, b1b);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ---- merge the consumer warps' states in shared memory (reusing the ring)
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers) : "memory");  // ring fully consumed
    float* mrg = reinterpret_cast<float*>(smem);
    float* wm = mrg + cw * (2 * kHeadsPerCta + kHeadsPerCta * D);
    float* wl = wm + kHeadsPerCta;
    float* wo = wl + kHeadsPerCta;
    if ((lane & 3) == 0) {
      wm[r_lo] = m_lo;
      wm[r_lo + 8] = m_hi;
      wl[r_lo] = l_lo;
      wl[r_lo + 8] = l_hi;
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      wo[r_lo * D + n * 8 + cpair] = o[n][0];
      wo[r_lo * D + n * 8 + cpair + 1] = o[n][1];
      wo[(r_lo + 8) * D + n * 8 + cpair] = o[n][2];
      wo[(r_lo + 8) * D + n * 8 + cpair + 1] = o[n][3];
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers) : "memory");
    const int tid = threadIdx.x - 32;
    const size_t ws_row0 = (static_cast<size_t>(b) * p.Hq + h0) * p.num_splits + split;
    for (int idx = tid; idx < nh * D; idx += 32 * kConsumers) {
      const int g = idx / D, t = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w)
        M = fmaxf(M, mrg[w * (2 * kHeadsPerCta + kHeadsPerCta * D) + g]);
      float acc = 0.f, lsum = 0.f;
      if (M != -INFINITY) {
        const float Ms = M * scale2;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) {
          const float* base = mrg + w * (2 * kHeadsPerCta + kHeadsPerCta * D);
          const float f = ex2_approx(fmaf(base[g], scale2, -Ms));
          lsum += base[kHeadsPerCta + g] * f;
          acc += base[2 * kHeadsPerCta + g * D + t] * f;
        }
      }
      const size_t wr = ws_row0 + static_cast<size_t>(g) * p.num_splits;
      const bool seen = lsum > 0.f;
      p.ws_o[wr * D + t] = seen ? acc / lsum : 0.f;
      if (t == 0) p.ws_lse[wr] = seen ? fmaf(M, p.scale, logf(lsum)) : -INFINITY;
    }
  }
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    // let copies already issued land before the shared memory is released
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) {
    }
  }
}

// Head dimension 256.  One accumulator tile of 16 query heads x 256 columns
// is 128 fp32 registers a thread, too many next to the rest of the state, so
// the two consumer warps both walk every page of the split: each forms
// S = Q K^T over the full head dimension (the same numbers in both, so the
// two online-softmax states stay identical) and keeps its own half of O,
// columns 128 w .. 128 w + 127.  Q fragments are read from shared memory page
// by page (64 registers saved).  A ring slot is released once both warps have
// read it.  Pages in flight per SM: two CTAs x 6 slots x 16 KB.
constexpr int kStages256 = 6;
constexpr int kQPitch256 = 256 * 2 + 16;  // bytes per staged query row (16-byte skew)

struct Dec256 {
  static constexpr int kAtoms = 4;
  static constexpr int kBoxBytes = kPage * 128;
  static constexpr int kSliceBytes = kAtoms * kBoxBytes;
  static constexpr int kStageBytes = 2 * kSliceBytes;
  static constexpr int kRingBytes = kStages256 * kStageBytes;
  static constexpr int kOffQ = kRingBytes;
  static constexpr int kOffBar = kOffQ + kHeadsPerCta * kQPitch256;
  static constexpr int kSmemBytes = kOffBar + 2 * kStages256 * 8 + 1024;
};

__global__ void __launch_bounds__(kDecThreads, 2)
    attn_decode_split256_kernel(const __grid_constant__ CUtensorMap tmK,
                                const __grid_constant__ CUtensorMap tmV, const DecParams p) {
  using C = Dec256;
  constexpr int D = 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* empty = full + kStages256;
  uint8_t* sq = smem + C::kOffQ;
  __shared__ int abort_flag_s;
  volatile int* abort_flag = &abort_flag_s;

  const int split = blockIdx.x;
  const int hkv = blockIdx.y / p.n_hchunks;
  const int hchunk = blockIdx.y % p.n_hchunks;
  // Launched as a programmatic dependent of the order kernel: the launch
  // overlaps it, and this waits for its result.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = p.order[blockIdx.z];
  const int g0 = hchunk * kHeadsPerCta;
  const int nh = min(kHeadsPerCta, p.G - g0);
  const int h0 = hkv * p.G + g0;

  int L = p.seqlens[b];
  if (L < 0 || L > p.max_pages * kPage) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusBadInput);
    L = max(0, min(L, p.max_pages * kPage));
  }
  const int np = (L + kPage - 1) / kPage;
  const int pps = (np + p.num_splits - 1) / p.num_splits;
  const int pg0 = min(split * pps, np);
  const int pg1 = min(pg0 + pps, np);
  const int npg = pg1 - pg0;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    abort_flag_s = 0;
    for (int s = 0; s < kStages256; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers);
    }
    fence_mbar_init();
  }
  // The served query heads' rows (16 x 256 bf16, rows past nh zero).
  {
    const __nv_bfloat16* qb = p.q + (static_cast<size_t>(b) * p.Hq + h0) * D;
    for (int idx = threadIdx.x; idx < kHeadsPerCta * (D / 8); idx += kDecThreads) {
      const int r = idx / (D / 8), c8 = idx % (D / 8);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (r < nh) v = *reinterpret_cast<const uint4*>(qb + static_cast<size_t>(r) * D + c8 * 8);
      *reinterpret_cast<uint4*>(sq + r * kQPitch256 + c8 * 16) = v;
    }
  }
  __syncthreads();

  if (warp == 0) {
    // ============================================================ producer
    if (lane == 0 && npg > 0) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const int* row = p.page_table + static_cast<size_t>(b) * p.max_pages;
      int page_next = row[pg0];  // each page index read one page ahead of its loads
      for (int i = 0; i < npg; ++i) {
        const int s = i % kStages256;
        int page = page_next;
        if (i + 1 < npg) page_next = row[pg0 + i + 1];
        if (!mbar_wait(&empty[s], ((i / kStages256) & 1) ^ 1, abort_flag, p.wait_limit_ns)) {
          atomicOr(p.status, kStatusTimeout);
          *abort_flag = 1;
          break;
        }
        if (page < 0 || page >= p.num_pages) {
          atomicOr(p.status, kStatusBadInput);
          page = p.num_pages;  // past the pool: the copy reads zeros
        }
        uint8_t* st = smem + s * C::kStageBytes;
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a) {
          tma_load_4d(st + a * C::kBoxBytes, &tmK, &full[s], a * 64, hkv, 0, page);
          tma_load_4d(st + C::kSliceBytes + a * C::kBoxBytes, &tmV, &full[s], a * 64, hkv, 0, page);
        }
      }
    }
    __syncwarp();
  } else {
    // ============================================================ consumers
    const int half = warp - 1;        // the O columns this warp keeps: 128 half ..
    const int r_lo = lane >> 2;
    const int cpair = (lane & 3) * 2;
    const int mi = lane >> 3, rr8 = lane & 7;
    // ldmatrix rows of the query fragments: matrix mi holds rows 8 (mi & 1) ..,
    // columns 8 (mi >> 1) .. of each 16 x 16 block.
    const uint32_t qrow = smem_addr(sq) + (rr8 + ((mi & 1) ? 8 : 0)) * kQPitch256 +
                          ((mi & 2) ? 16 : 0);
    float o[D / 16][4];
#pragma unroll
    for (int n = 0; n < D / 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
    const float scale2 = p.scale2;
    bool ok = true;
    for (int i = 0; i < npg; ++i) {
      const int s = i % kStages256;
      ok = mbar_wait(&full[s], (i / kStages256) & 1, abort_flag, p.wait_limit_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) {
          atomicOr(p.status, kStatusTimeout);
          *abort_flag = 1;
        }
        break;
      }
      const uint32_t kst = smem_addr(smem + s * C::kStageBytes);
      const uint32_t vst = kst + C::kSliceBytes;
      // ---- S[16 heads x 16 tokens] = Q K^T over all 256 columns
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t qa[4];
        ldsm_x4(qrow + kk * 32, qa[0], qa[1], qa[2], qa[3]);
        const int tok = rr8 + ((mi & 2) ? 8 : 0);
        const int e = kk * 16 + ((mi & 1) ? 8 : 0);
        uint32_t b00, b01, b10, b11;
        ldsm_x4(kst + (e / 64) * C::kBoxBytes + swz(tok, e % 64), b00, b01, b10, b11);
        mma16816(sc[0], qa, b00, b01);
        mma16816(sc[1], qa, b10, b11);
      }
      const int tok_base = (pg0 + i) * kPage;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (tok_base + nt * 8 + cpair + (e & 1) >= L) sc[nt][e] = -INFINITY;
      float mx_lo = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float mx_hi = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
      const float ms_lo = (mn_lo == -INFINITY) ? 0.f : mn_lo * scale2;
      const float ms_hi = (mn_hi == -INFINITY) ? 0.f : mn_hi * scale2;
      const float a_lo = ex2_approx(fmaf(m_lo, scale2, -ms_lo));
      const float a_hi = ex2_approx(fmaf(m_hi, scale2, -ms_hi));
      m_lo = mn_lo;
      m_hi = mn_hi;
      uint32_t pa[4];
      float ps_lo = 0.f, ps_hi = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float p0 = ex2_approx(fmaf(sc[nt][0], scale2, -ms_lo));
        const float p1 = ex2_approx(fmaf(sc[nt][1], scale2, -ms_lo));
        const float p2 = ex2_approx(fmaf(sc[nt][2], scale2, -ms_hi));
        const float p3 = ex2_approx(fmaf(sc[nt][3], scale2, -ms_hi));
        ps_lo += p0 + p1;
        ps_hi += p2 + p3;
        pa[nt * 2 + 0] = pack_bf16x2(p0, p1);
        pa[nt * 2 + 1] = pack_bf16x2(p2, p3);
      }
      l_lo = l_lo * a_lo + ps_lo;
      l_hi = l_hi * a_hi + ps_hi;
      // ---- this warp's half of O = alpha O + P V
#pragma unroll
      for (int n = 0; n < D / 16; ++n) {
        o[n][0] *= a_lo;
        o[n][1] *= a_lo;
        o[n][2] *= a_hi;
        o[n][3] *= a_hi;
      }
#pragma unroll
      for (int n2 = 0; n2 < D / 32; ++n2) {
        const int tok = rr8 + ((mi & 1) ? 8 : 0);
        const int e = half * (D / 2) + n2 * 16 + ((mi & 2) ? 8 : 0);
        uint32_t b0a, b1a, b0b, b1b;
        ldsm_x4_t(vst + (e / 64) * C::kBoxBytes + swz(tok, e % 64), b0a, b1a, b0b, b1b);
        mma16816(o[2 * n2], pa, b0a, b1a);
        mma16816(o[2 * n2 + 1], pa, b0b, b1b);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // ---- the split's normalised half of O and, from warp 1, its LSE
    if (ok) {
      l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
      l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
      l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
      l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
      const size_t ws_row0 = (static_cast<size_t>(b) * p.Hq + h0) * p.num_splits + split;
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int g = r_lo + 8 * hr;
        if (g >= nh) continue;
        const float l = hr ? l_hi : l_lo, m = hr ? m_hi : m_lo;
        const bool seen = l > 0.f;
        const float inv = seen ? 1.f / l : 0.f;
        const size_t wr = ws_row0 + static_cast<size_t>(g) * p.num_splits;
        float* dst = p.ws_o + wr * D + half * (D / 2);
#pragma unroll
        for (int n = 0; n < D / 16; ++n) {
          dst[n * 8 + cpair] = o[n][2 * hr] * inv;
          dst[n * 8 + cpair + 1] = o[n][2 * hr + 1] * inv;
        }
        if (half == 0 && (lane & 3) == 0)
          p.ws_lse[wr] = seen ? fmaf(m, p.scale, logf(l)) : -INFINITY;
      }
    }
  }
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    // let copies already issued land before the shared memory is released
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) {
    }
  }
}

// Merge of the split partials, ascending split order (deterministic).
template <int D>
__global__ void __launch_bounds__(D)
    attn_decode_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                               __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                               int num_splits, const float* __restrict__ sink, int Hq) {
  // Launched as a programmatic dependent of the split kernel: its launch
  // overlaps the split's tail, and this waits for the split's results.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const size_t row = blockIdx.x;  // b * Hq + h
  const float* ls = ws_lse + row * num_splits;
  // A logit sink joins the merge as one more denominator term with no output
  // ("TileLang tutorial, ch.15", section 4.6), against M = max(sink, lse_s).
  const float sg = sink ? sink[row % static_cast<size_t>(Hq)] : -INFINITY;
  float M = sg;
  for (int s = 0; s < num_splits; ++s) M = fmaxf(M, ls[s]);
  const int t = threadIdx.x;
  if (M == -INFINITY) {
    o[row * D + t] = __float2bfloat16(0.f);
    if (lse && t == 0) lse[row] = -INFINITY;
    return;
  }
  float wsum = (sg == -INFINITY) ? 0.f : expf(sg - M), acc = 0.f;
  for (int s = 0; s < num_splits; ++s) {
    const float w = expf(ls[s] - M);
    wsum += w;
    acc += w * ws_o[(row * num_splits + s) * D + t];
  }
  o[row * D + t] = __float2bfloat16(acc / wsum);
  if (lse && t == 0) lse[row] = M + logf(wsum);
}

// The merge, launched so that it may start while the split kernel drains
// (programmatic stream serialization; the kernel's griddepcontrol.wait
// keeps its reads after the split's writes).
template <int D>
cudaError_t launch_combine(const DecodeLaunch& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.Hq);
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_decode_combine_kernel<D>,
                            static_cast<const float*>(a.ws_o), static_cast<const float*>(a.ws_lse),
                            static_cast<__nv_bfloat16*>(a.o), a.lse, a.num_splits, a.sink, a.Hq);
}

// The request order, then the split kernel as its programmatic dependent.
template <typename Kernel>
cudaError_t launch_ordered(const DecodeLaunch& a, Kernel kernel, dim3 grid, size_t smem,
                           const DecParams& p, cudaStream_t stream) {
  attn_decode_order_kernel<<<1, kOrderThreads, 0, stream>>>(a.seqlens, a.B, a.max_pages, a.order);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a.tmK, a.tmV, p);
}

template <int D>
cudaError_t launch_dec(const DecodeLaunch& a, cudaStream_t stream) {
  using C = DecCfg<D>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_decode_split_kernel<D>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  DecParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.page_table = a.page_table;
  p.seqlens = a.seqlens;
  p.ws_o = a.ws_o;
  p.ws_lse = a.ws_lse;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.Hq / a.Hkv;
  p.n_hchunks = (p.G + kHeadsPerCta - 1) / kHeadsPerCta;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.num_splits = a.num_splits;
  p.scale = a.scale;
  p.scale2 = a.scale * kLog2eDec;
  p.wait_limit_ns = kWaitLimitNs;
  p.status = a.status;
  dim3 grid(a.num_splits, a.Hkv * p.n_hchunks, a.B);
  p.order = a.order;
  cudaError_t e =
      launch_ordered(a, attn_decode_split_kernel<D>, grid, C::kSmemBytes, p, stream);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_combine<D>(a, stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}


cudaError_t launch_dec256(const DecodeLaunch& a, cudaStream_t stream) {
  using C = Dec256;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_decode_split256_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  DecParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.page_table = a.page_table;
  p.seqlens = a.seqlens;
  p.ws_o = a.ws_o;
  p.ws_lse = a.ws_lse;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.Hq / a.Hkv;
  p.n_hchunks = (p.G + kHeadsPerCta - 1) / kHeadsPerCta;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.num_splits = a.num_splits;
  p.scale = a.scale;
  p.scale2 = a.scale * kLog2eDec;
  p.wait_limit_ns = kWaitLimitNs;
  p.status = a.status;
  dim3 grid(a.num_splits, a.Hkv * p.n_hchunks, a.B);
  p.order = a.order;
  cudaError_t e = launch_ordered(a, attn_decode_split256_kernel, grid, C::kSmemBytes, p, stream);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_combine<256>(a, stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_decode(const DecodeLaunch& a, cudaStream_t stream) {
  if (a.d == 128) return launch_dec<128>(a, stream);
  if (a.d == 64) return launch_dec<64>(a, stream);
  if (a.d == 256) return launch_dec256(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
