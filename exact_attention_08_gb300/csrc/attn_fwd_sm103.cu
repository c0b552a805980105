// Exact attention forward for sm_103a: tcgen05 MMAs with accumulators in
// tensor memory, TMA-fed K/V ring, online softmax fused between the two
// matrix products.
//
// One CTA owns 256 consecutive query rows of one (batch or sequence, query
// head): two 128-row Q tiles, resident in shared memory for the whole key
// loop (the FA-2 order: query tiles in the grid, key/value tiles in the inner
// loop; "TileLang in practice: FlashAttention forward kernel", sections 3.1
// and 5; "TileLang tutorial, ch.15 Operators: Attention", section 2.5).
// Keys and values stream through a ring of 128-key tiles.
//
// Warp roles (12 warps, three warpgroups):
//   warps 0-3   softmax for Q tile 0 (thread r owns query row r: TMEM lane r),
//               and its O epilogue (direct stores of each thread's row)
//   warps 4-7   softmax for Q tile 1
//   warp  8     TMA producer (Q tiles through three slots, the K/V ring);
//               allocates TMEM
//   warp  9     MMA issuer (whole warp, one elected lane issues)
//   warp  10    builds the dense item order of causal packed calls at start
//   warps 10-11 otherwise idle (the register split needs whole warpgroups)
// Tensor memory (512 columns): S_i = Q_i K^T at columns [128 i, 128 i + 128)
// (fp32), O_i at [256 + D i, 256 + D i + D) (fp32).  The softmax writes the
// probabilities P_i back over the first 64 columns of S_i as packed bf16
// pairs (32 key columns at a time, over scores it has already read), and the
// second product O_i += P_i V reads P_i straight from tensor memory, so
// neither S nor P ever leaves the SM.  P_i is published in two halves: the
// tensor core starts O_i += P_i V on keys 0..63 while the softmax still forms
// keys 64..127.
//
// MMA issue order per key tile j:  O_0 += P_0(j-1) V(j-1), S_0 = Q_0 K(j)^T,
// O_1 += P_1(j-1) V(j-1), S_1 = Q_1 K(j)^T.  While warpgroup 0 turns S_0(j)
// into P_0(j), the tensor core runs O_1(j-1) and S_1(j), and vice versa, so
// the exponentials of one tile overlap the matrix products of the other.
//
// Online softmax per row (ch.15 section 2.3): raw row maximum m (the scale is
// applied inside the exponent, ch.15 section 3.2: max(s x) = s max(x)),
// exponent base 2 with log2(e) folded into the scale, running sum l, final
// O / l, LSE = m * scale + ln(l).  The rescale of O and l by
// exp2((m_old - m_new) * scale * log2 e) is applied only when the maximum grows
// by more than 8 in log2 units; otherwise the stale maximum is kept, which is
// exact (any common shift cancels between O and l, ch.15 section 2.4) and
// keeps every probability below 2^8.  A maximum of -inf (no visible key yet)
// is replaced by 0 in the exponent (check_inf, ch.15 section 5.1(1)); a row
// that never sees a key returns O = 0 and LSE = -inf (section 5.1(2)).
//
// Masks (ch.15 sections 3.4, 5.2): tiles that no row of a Q tile can see are
// never loaded (causal upper bound, window lower bound, sink tiles kept);
// tiles every row sees in full skip the mask; only boundary tiles compare
// key indices, in registers after the tensor-memory load.
#include "attn_internal.h"
#include "sm103_ptx.cuh"

#include <cuda_bf16.h>
#include <algorithm>
#include <climits>
#include <mutex>

namespace attn {
namespace {

using namespace ptx;

constexpr int kBM = 128;       // query rows per Q tile (= TMEM lanes)
constexpr int kQT = 2;         // Q tiles per work item
constexpr int kQSlots = 3;     // Q tile buffers in shared memory
constexpr int kBN = 128;       // keys per K/V tile
constexpr int kPage = 16;      // keys per page of a paged cache
constexpr int kPagesPerTile = kBN / kPage;
constexpr int kThreads = 384;  // 12 warps
constexpr int kRegsSoftmax = 192;
constexpr int kRegsOther = 120;
// Registers the three warpgroups hold after setmaxnreg; must not exceed what
// the block is launched with (checked on the host before every launch).
constexpr int kRegsSplit = 2 * 128 * kRegsSoftmax + 128 * kRegsOther;
static_assert(kRegsSplit <= kThreads * 168, "register split");
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpTable = 10;  // builds the dense item order of packed calls, then locates items
// Item records in flight between the locating warp and the roles, and the
// arrivals that free one: the producer and MMA warps, the eight softmax warps.
constexpr int kRecSlots = 4;
constexpr int kRecReaders = 10;
constexpr int kPrefetch = 2;  // key/value tiles warmed in L2 ahead of their load
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;
// Lower visibility bound when there is no window: far below every key index,
// yet chunk offsets (at most a few hundred) can be subtracted without overflow.
constexpr int kNoLowerBound = -(1 << 29);

template <int D>
struct Cfg {
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kTileBytes = kBM * D * 2;  // 128 rows x D bf16 (Q, K, V and O tiles alike)
  static constexpr int kAtoms = D / 64;           // 128-byte swizzle atoms per row
  static constexpr int kAtomBytes = 128 * 128;    // one atom column of a tile: 128 rows x 128 B
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQSlots * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  // q_full[3], q_empty[3], k_full[S], v_full[S], step[S], s_full[2], p_half[2], p_ready[2],
  // o_done[2], drain, rec_full[R], rec_empty[R]
  static constexpr int kNumBars = 2 * kQSlots + 3 * kStages + 4 * kQT + 1 + 2 * kRecSlots;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 2 * kBN;
};

// Division of a non-negative 31-bit integer by a fixed divisor d >= 1 with a
// multiplier computed once on the host (Granlund and Montgomery, "Division
// by invariant integers using multiplication", 1994: l = ceil(log2 d),
// m = floor(2^32 (2^l - d) / d) + 1, n / d = (mulhi(n, m) + n) >> l; the sum
// cannot overflow for n < 2^31).  Item decoding divides by the head count,
// the batch and the pair count on every item of every role, and a plain
// integer division there costs tens of instructions.
struct FastDiv {
  uint32_t d, m, l;
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d;
  f.l = 0;
  while ((1ull << f.l) < d) ++f.l;
  f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << f.l) - d)) / d + 1);
  return f;
}

__device__ __forceinline__ int fdiv(int n, const FastDiv& f) {
  const uint32_t u = static_cast<uint32_t>(n);
  return static_cast<int>((__umulhi(u, f.m) + u) >> f.l);
}

struct Params {
  __nv_bfloat16* o;
  long long o_sb, o_ss, o_sh;  // O strides (elements): batch, row, head; d contiguous
  int o_v8;                    // every O row starts on 32 bytes: 32-byte stores
  float* lse;
  const float* sink;  // logit sink per query head [Hq], or null
  const int* cu_q;
  const int* cu_k;
  const int* page_table;  // paged K/V: [B, max_pages] physical pages, or null
  const int* seqlens_k;   // paged K/V: key count of every sequence [B]
  int max_pages, num_pages;
  int B, Hq, Hkv, Sq, Skv, total_q;
  int num_qpairs, num_items;
  FastDiv div_hq, div_b, div_qp, div_group;  // by Hq, B, num_qpairs, Hq / Hkv
  float scale, scale2;
  int causal, window, n_sink;
  uint64_t wait_limit_ns;
  int* status;
};

// Rows [qa, qb) of one Q tile (sequence-relative) and the extreme visible-key
// bounds over those rows: key k is visible to row q iff k <= hi(q) and, with a
// window, (k > lo(q) or k < n_sink).
struct TileMask {
  int qa, qb;
  int hi_min, hi_max;  // hi(qa), hi(qb - 1)
  int lo_min, lo_max;  // lo(qa), lo(qb - 1)
};

__device__ __forceinline__ TileMask make_mask(int qa, int Lq, int Lk, int off, int causal,
                                              int window) {
  TileMask m;
  m.qa = qa;
  m.qb = min(qa + kBM, Lq);
  const int last = max(m.qb - 1, qa);
  m.hi_min = causal ? min(qa + off, Lk - 1) : Lk - 1;
  m.hi_max = causal ? min(last + off, Lk - 1) : Lk - 1;
  m.lo_min = (window > 0) ? qa + off - window : kNoLowerBound;
  m.lo_max = (window > 0) ? last + off - window : kNoLowerBound;
  return m;
}

// The key tiles a Q tile touches, as two ranges: tile j is active iff
// j <= hi and (j >= lo or j < sinkT), sinkT = ceil(n_sink / kBN) the tiles
// holding sink keys.  The same set as "does any row of the tile see any key
// of tile j": hi is the last tile holding a key at or below the largest
// causal bound (and below Lk), lo the first tile holding a key above the
// smallest window bound.
struct TileRange {
  int lo, hi;
};

__device__ __forceinline__ TileRange tile_range(const TileMask& m, int Lk, int window) {
  TileRange r;
  if (m.qb <= m.qa || m.hi_max < 0 || Lk <= 0) {
    r.lo = 0;
    r.hi = -1;
    return r;
  }
  r.hi = min((Lk - 1) / kBN, m.hi_max / kBN);
  if (window <= 0)
    r.lo = 0;
  else if (m.lo_min >= Lk - 1)
    r.lo = r.hi + 1;  // only sink keys are visible
  else
    r.lo = (m.lo_min < 0) ? 0 : (m.lo_min + 1) / kBN;
  return r;
}

__device__ __forceinline__ bool in_range(const TileRange& r, int j, int sinkT) {
  return j <= r.hi && (j >= r.lo || j < sinkT);
}

// The first active tile of a range at or after c (INT_MAX: none): the sink
// tiles, then the window's tiles from r.lo on.  Loops over a Q tile's keys
// step from one active tile to the next, so a window far from the sink costs
// no iterations over the tiles between.
__device__ __forceinline__ int next_in_range(const TileRange& r, int c, int sinkT) {
  const int n = (c < sinkT) ? c : max(c, r.lo);
  return n <= r.hi ? n : INT_MAX;
}

// The first tile at or after c active for either Q tile of an item.
__device__ __forceinline__ int next_in_pair(const TileRange& r0, const TileRange& r1, int c,
                                            int sinkT) {
  return min(next_in_range(r0, c, sinkT), next_in_range(r1, c, sinkT));
}

// Does every row of the tile see every key of key tile j (no mask needed)?
__device__ __forceinline__ bool tile_interior(const TileMask& m, int j, int window, int n_sink) {
  const int ka = j * kBN, kb1 = ka + kBN - 1;
  if (kb1 > m.hi_min) return false;  // hi_min <= Lk - 1 also rules out the ragged tail
  if (window > 0 && !(ka > m.lo_max || kb1 < n_sink)) return false;
  return true;
}

__device__ __forceinline__ void reg_fence(uint32_t& r) { asm volatile("" : "+r"(r)); }

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void fail(int* status, volatile int* abort_flag) {
  atomicOr(status, kStatusTimeout);
  *abort_flag = 1;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}

// Packed pairs of fp32 (one 64-bit register, two lanes of arithmetic per
// instruction).
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Maximum of 32 scores (and a running value), as a shallow tree.
__device__ __forceinline__ float max32(const uint32_t* v, float run) {
  float a[11];
#pragma unroll
  for (int t = 0; t < 10; ++t)
    a[t] = max3(__uint_as_float(v[3 * t]), __uint_as_float(v[3 * t + 1]),
                __uint_as_float(v[3 * t + 2]));
  a[10] = max3(__uint_as_float(v[30]), __uint_as_float(v[31]), run);
  const float b0 = max3(a[0], a[1], a[2]), b1 = max3(a[3], a[4], a[5]);
  const float b2 = max3(a[6], a[7], a[8]), b3 = fmaxf(a[9], a[10]);
  return max3(b0, b1, fmaxf(b2, b3));
}

// Bits [0, n) of a 32-bit word, n clamped to [0, 32].
__device__ __forceinline__ uint32_t low_bits(int n) {
  return n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : (1u << n) - 1u);
}

// The keys of a 32-key chunk a row may see, as a bit mask: column c is key
// kc0 + c, visible iff c <= lim_hi and (c > lim_lo or c < lim_sink), all
// limits relative to kc0.
__device__ __forceinline__ uint32_t visible32(int lim_hi, int lim_lo, int lim_sink) {
  const int lo1 = max(lim_lo, -1) + 1;  // first column above the window's lower bound
  return low_bits(lim_hi + 1) & (~low_bits(lo1) | low_bits(lim_sink));
}

// Sets the scores of the keys a row may not see to -inf (one bit test and
// one select per score); nothing to do when the whole warp sees the chunk.
__device__ __forceinline__ void mask32(uint32_t* v, int lim_hi, int lim_lo, int lim_sink) {
  const uint32_t vis = visible32(lim_hi, lim_lo, lim_sink);
  if (__all_sync(0xffffffffu, vis == 0xffffffffu)) return;
#pragma unroll
  for (int c = 0; c < 32; ++c)
    if (!(vis & (1u << c))) v[c] = __float_as_uint(-INFINITY);
}

// Exponentials of 32 scores: p = 2^(s * scale2 - ms), accumulated into the
// packed running sums and packed to bf16 pairs in pk[16].
__device__ __forceinline__ void exp32(const uint32_t* v, uint64_t sc2, uint64_t nms,
                                      uint64_t& sum_a, uint64_t& sum_b, uint32_t* pk) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const uint64_t x = f2_fma(f2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sc2,
                              nms);
    float x0, x1;
    f2_split(x, x0, x1);
    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    if (e & 1)
      sum_b = f2_add(sum_b, f2(p0, p1));
    else
      sum_a = f2_add(sum_a, f2(p0, p1));
    pk[e] = pack_bf16x2(p0, p1);
  }
}

// Work item k (a pair of Q tiles of one (batch or sequence, query head)):
// its coordinates, lengths, masks and active key-tile ranges.
struct Work {
  int bseq, h, hk, q0, Lq, Lk, off, q_base, k_base, b_coord, lastT;
  TileMask m0, m1;
  TileRange r0, r1;
};

// Causal packed calls (varlen, paged) with up to kTabMaxSeq sequences and
// kTabMaxLev query pairs per sequence walk a dense item order: only the
// (sequence, query pair) combinations that hold query rows, level by level
// from the last query pair down (causal work grows with the pair index), the
// sequences of a level in decreasing order of their pair count.  In the
// sparse order, a level of short sequences is mostly empty items, and the
// persistent CTAs that drew them ended up with less work than the others
// (measured on 8 sequences of 900-3198 rows: key steps per CTA 112-179
// against a mean of 147).  One warp builds the table at kernel start.
constexpr int kTabMaxSeq = 256;
constexpr int kTabMaxLev = 64;
// Query blocks against a paged cache (chunked prefill, speculative decoding)
// read far more keys than they have queries, so an item's cost follows its
// sequence's key count rather than its query pair: batches of up to
// kTabSortMax sequences are ordered by key count instead (longest first,
// each sequence's query pairs last first, its heads adjacent).
constexpr int kTabSortMax = 64;

struct ItemTable {
  int total;                       // items in the dense order (0: the table is not used)
  int lev_start[kTabMaxLev + 1];   // dense sequence slots before each level
  int hist[kTabMaxLev + 1];        // sequences by pair count (scratch of the build)
  short order[kTabMaxSeq];         // sequences, most query pairs first
};

// The query rows of packed sequence b, or -1 when its offsets are invalid
// (the same checks as locate_item).
template <bool kPagedKV>
__device__ __forceinline__ int packed_rows(const Params& p, int b) {
  const int a = p.cu_q[b], e = p.cu_q[b + 1];
  if (a < 0 || e < a || e > p.total_q || e - a > p.Sq) return -1;
  if (kPagedKV) {
    const int lk = p.seqlens_k[b];
    if (lk < 0 || lk > p.max_pages * kPage) return -1;
  } else {
    const int ka = p.cu_k[b], ke = p.cu_k[b + 1];
    if (ka < 0 || ke < ka) return -1;
  }
  return e - a;
}

// Builds the dense order (one warp).  Sequences with invalid offsets are
// reported and left out.
template <bool kPagedKV>
__device__ __forceinline__ void build_item_table(const Params& p, ItemTable& t, int lane) {
  if (kPagedKV && p.B <= kTabSortMax) {
    // by key tiles, ties by sequence index: hist[b] the key tiles of b and
    // lev_start[b + 1] its pairs, then order[rank] = b, hist[rank] its
    // pairs, and lev_start the running slot counts
    const int nlev = p.num_qpairs;
    int rk[2], npb[2];
    for (int i = 0; i < 2; ++i) {
      const int b = lane + 32 * i;
      if (b < p.B) {
        const int rows = packed_rows<kPagedKV>(p, b);
        if (rows < 0) atomicOr(p.status, kStatusBadInput);
        npb[i] = rows <= 0 ? 0 : min((rows + kQT * kBM - 1) / (kQT * kBM), nlev);
        t.hist[b] = rows < 0 ? 0 : (p.seqlens_k[b] + kBN - 1) / kBN;
      }
    }
    __syncwarp();
    for (int i = 0; i < 2; ++i) {
      const int b = lane + 32 * i;
      rk[i] = 0;
      if (b < p.B) {
        const int kb = t.hist[b];
        for (int c = 0; c < p.B; ++c) {
          const int kc = t.hist[c];
          rk[i] += (kc > kb || (kc == kb && c < b)) ? 1 : 0;
        }
      }
    }
    __syncwarp();
    for (int i = 0; i < 2; ++i) {
      const int b = lane + 32 * i;
      if (b < p.B) {
        t.order[rk[i]] = static_cast<short>(b);
        t.hist[rk[i]] = npb[i];
      }
    }
    __syncwarp();
    if (lane == 0) {
      t.lev_start[0] = 0;
      for (int r = 0; r < p.B; ++r) t.lev_start[r + 1] = t.lev_start[r] + t.hist[r];
      t.total = t.lev_start[p.B] * p.Hq;
    }
    __syncwarp();
    return;
  }
  const int nlev = p.num_qpairs;
  for (int l = lane; l <= nlev; l += 32) t.hist[l] = 0;
  __syncwarp();
  for (int b = lane; b < p.B; b += 32) {
    const int rows = packed_rows<kPagedKV>(p, b);
    if (rows < 0) atomicOr(p.status, kStatusBadInput);
    const int np = rows <= 0 ? 0 : min((rows + kQT * kBM - 1) / (kQT * kBM), nlev);
    atomicAdd(&t.hist[np], 1);
  }
  __syncwarp();
  if (lane == 0) {
    // hist[np] becomes the first slot of the sequences with np pairs (most
    // pairs first); level qp holds the sequences with more than qp pairs.
    int run = 0;
    for (int np = nlev; np >= 0; --np) {
      const int c = t.hist[np];
      t.hist[np] = run;
      run += c;
    }
    t.lev_start[0] = 0;
    for (int l = 0; l < nlev; ++l) {
      const int qp = nlev - 1 - l;
      t.lev_start[l + 1] = t.lev_start[l] + t.hist[qp];  // sequences with > qp pairs
    }
    t.total = t.lev_start[nlev] * p.Hq;
  }
  __syncwarp();
  for (int b = lane; b < p.B; b += 32) {
    const int rows = packed_rows<kPagedKV>(p, b);
    const int np = rows <= 0 ? 0 : min((rows + kQT * kBM - 1) / (kQT * kBM), nlev);
    t.order[atomicAdd(&t.hist[np], 1)] = static_cast<short>(b);
  }
  __syncwarp();
}

// Item order.  Without causal masking every item is the same work; the
// query pairs of one (batch, head) are consecutive, so CTAs streaming the
// same keys and values run together and share them through L2.  With
// causal masking the work of a pair grows with its index: the longest pairs
// of every head come first (for packed calls through the dense table when
// there is one).  Heads of one KV group are adjacent either way.
//
// What locating an item takes the item table or global memory (the
// sequence offsets) for; work_of derives the rest.
struct ItemLoc {
  int bseq, h, q0, Lq, Lk, q_base, k_base;
};

// Locates item k.  Returns false when it has no query rows or its sequence
// offsets are invalid (reported when report is set).
template <bool kPagedKV, bool kTable>
__device__ __forceinline__ bool locate_item(const Params& p, const ItemTable& tab, int k,
                                            ItemLoc& r, bool report) {
  int qp;
  if (kTable && kPagedKV && p.B <= kTabSortMax) {
    // the sequence rank r with lev_start[r] <= sl < lev_start[r + 1], its
    // query pairs last first
    const int sl = fdiv(k, p.div_hq);
    r.h = k - sl * p.Hq;
    int lo = 0, hi = p.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tab.lev_start[mid] <= sl)
        lo = mid;
      else
        hi = mid;
    }
    qp = tab.lev_start[lo + 1] - 1 - sl;
    r.bseq = tab.order[lo];
  } else if (kTable) {
    const int sl = fdiv(k, p.div_hq);
    r.h = k - sl * p.Hq;
    int lo = 0, hi = p.num_qpairs;  // the level l with lev_start[l] <= sl < lev_start[l + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tab.lev_start[mid] <= sl)
        lo = mid;
      else
        hi = mid;
    }
    qp = p.num_qpairs - 1 - lo;
    r.bseq = tab.order[sl - tab.lev_start[lo]];
  } else if (p.causal) {
    const int x = fdiv(k, p.div_hq), y = fdiv(x, p.div_b);
    r.h = k - x * p.Hq;
    r.bseq = x - y * p.B;
    qp = p.num_qpairs - 1 - y;
  } else {
    const int x = fdiv(k, p.div_qp), y = fdiv(x, p.div_hq);
    qp = k - x * p.num_qpairs;
    r.h = x - y * p.Hq;
    r.bseq = y;
  }
  if (kPagedKV) {
    // Packed queries against a paged cache: the sequence's keys are its
    // first seqlens_k[b] cache slots, reached through its page-table row.
    const int a = p.cu_q[r.bseq], e = p.cu_q[r.bseq + 1];
    const int lk = p.seqlens_k[r.bseq];
    if (a < 0 || e < a || e > p.total_q || e - a > p.Sq || lk < 0 || lk > p.max_pages * kPage) {
      if (report) atomicOr(p.status, kStatusBadInput);
      return false;
    }
    r.Lq = e - a;
    r.Lk = lk;
    r.q_base = a;
    r.k_base = 0;
  } else if (p.cu_q != nullptr) {
    const int a = p.cu_q[r.bseq], e = p.cu_q[r.bseq + 1];
    const int ka = p.cu_k[r.bseq], ke = p.cu_k[r.bseq + 1];
    if (a < 0 || e < a || e > p.total_q || ka < 0 || ke < ka || e - a > p.Sq) {
      if (report) atomicOr(p.status, kStatusBadInput);
      return false;
    }
    r.Lq = e - a;
    r.Lk = ke - ka;
    r.q_base = a;
    r.k_base = ka;
  } else {
    r.Lq = p.Sq;
    r.Lk = p.Skv;
    r.q_base = 0;
    r.k_base = 0;
  }
  r.q0 = qp * (kQT * kBM);
  return r.q0 < r.Lq;
}

// Coordinates, masks and active key-tile ranges of a located item.
template <bool kPagedKV>
__device__ __forceinline__ void work_of(const Params& p, const ItemLoc& r, Work& w) {
  w.bseq = r.bseq;
  w.h = r.h;
  w.q0 = r.q0;
  w.Lq = r.Lq;
  w.Lk = r.Lk;
  w.q_base = r.q_base;
  w.k_base = r.k_base;
  w.b_coord = (kPagedKV || p.cu_q != nullptr) ? 0 : r.bseq;
  w.off = w.Lk - w.Lq;
  w.hk = fdiv(w.h, p.div_group);
  w.m0 = make_mask(w.q0, w.Lq, w.Lk, w.off, p.causal, p.window);
  w.m1 = make_mask(w.q0 + kBM, w.Lq, w.Lk, w.off, p.causal, p.window);
  w.r0 = tile_range(w.m0, w.Lk, p.window);
  w.r1 = tile_range(w.m1, w.Lk, p.window);
  w.lastT = max(w.r0.hi, w.r1.hi);  // last key tile any row touches (-1: none)
}

// Number of active key tiles of a range.
__device__ __forceinline__ int range_count(const TileRange& r, int sinkT) {
  if (r.hi < 0) return 0;
  return min(sinkT, r.hi + 1) + max(0, r.hi - max(r.lo, sinkT) + 1);
}

// An item as the locating warp hands it to the other roles: its decoding
// and the active key-tile counts of its two Q tiles.  live = 0 marks the end
// of a CTA's items.
struct ItemRec {
  Work w;
  int count0, count1;
  int live;
};

// The n-th item of this CTA: items are dealt out in bands of gridDim.x, every
// other band in reverse CTA order, so that with the longest items first the
// CTAs' totals even out.  -1 when the CTA has no n-th item.
__device__ __forceinline__ int item_of(int n, int num_items) {
  const int G = gridDim.x;
  const int pos = (n & 1) ? (G - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  const long long k = static_cast<long long>(n) * G + pos;
  return k < num_items ? static_cast<int>(k) : -1;
}

template <int D, bool kPagedKV, bool kTable>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const Params p) {
  using C = Cfg<D>;
  constexpr int ST = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;                 // [kQSlots]: the Q tile in slot s has landed
  uint64_t* q_empty = q_full + kQSlots;    // [kQSlots]: every S of the Q tile in slot s is done
  uint64_t* k_full = q_empty + kQSlots;
  uint64_t* v_full = k_full + ST;
  uint64_t* step = v_full + ST;  // step[u % ST]: every product of key step u is done
  uint64_t* s_full = step + ST;
  uint64_t* p_half = s_full + kQT;   // [2]: P_i of keys 0..63 written
  uint64_t* p_ready = p_half + kQT;  // [2]: all of P_i written
  uint64_t* o_done = p_ready + kQT;
  uint64_t* drain = o_done + kQT;
  uint64_t* rec_full = drain + 1;              // [kRecSlots]: item record written
  uint64_t* rec_empty = rec_full + kRecSlots;  // [kRecSlots]: every role is done with it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rec_empty + kRecSlots);
  __shared__ int abort_flag_s;
  volatile int* abort_flag = &abort_flag_s;
  __shared__ ItemTable tab;
  __shared__ ItemRec recs[kRecSlots];

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int sinkT = (p.window > 0 && p.n_sink > 0) ? (p.n_sink + kBN - 1) / kBN : 0;

  // ---------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    abort_flag_s = 0;
    for (int s = 0; s < kQSlots; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < ST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&step[s], 1);
    }
    for (int i = 0; i < kQT; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_half[i], 128);
      mbar_init(&p_ready[i], 128);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(drain, 1);
    for (int s = 0; s < kRecSlots; ++s) {
      mbar_init(&rec_full[s], 1);
      mbar_init(&rec_empty[s], kRecReaders);
    }
    fence_mbar_init();
  }
  if (warp == kWarpLoad) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  if (kTable && warp == kWarpTable) build_item_table<kPagedKV>(p, tab, lane);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int num_items = kTable ? tab.total : p.num_items;
  // Waits, for a whole warp, until record c of this CTA's item sequence is
  // out (false when the wait gave up); the caller reads recs[c % kRecSlots]
  // and frees it with release_item once it is done.
  auto take_item = [&](int c) -> bool {
    return mbar_wait_warp(&rec_full[c % kRecSlots], (c / kRecSlots) & 1, abort_flag,
                          p.wait_limit_ns);
  };
  auto release_item = [&](int c) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&rec_empty[c % kRecSlots]);
  };

  // The CTA is persistent: one warp locates its items (item_of, then the
  // table or the sequence offsets) ahead of the others and hands them over
  // as records in a ring of kRecSlots; every role takes the same records in
  // the same order, and its ring, barrier-phase and step counters carry over
  // from one item to the next.
  //
  // Q tiles.  The g-th Q tile this CTA loads (two per item with key tiles,
  // tile 0 then tile 1) goes to slot g % 3; the slot is refilled once every
  // S product of its previous tile, g - 3, is done (q_empty).  Tile 0 of an
  // item therefore reuses the slot of the item two back and is loaded about
  // one item ahead; tile 1 reuses the slot of tile 0 of the item before,
  // free as soon as that item's last S_0 is done.
  //
  // Key steps.  Ring tile u (the u-th active key tile loaded by this CTA,
  // counted over all its items) is key step u of the MMA issuer: the
  // products P V of the tile before it (whichever item that tile belongs
  // to), S_0(u) and S_1(u), then one commit on step[u % ST].  So K(u) is free
  // once step u is done and V(u) once step u + 1 is.  An item change is an
  // ordinary key step: the last P V of the old item and the first S of the
  // new one share it, and the old item's O epilogue runs while the tensor
  // core works on the new item's S.  After the last item a final step holds
  // only the outstanding products P V.
  //
  // Register budget: the block is launched with 168 registers a thread (three
  // warps share SMSP 0).  Each warpgroup changes its budget at the head of
  // the branch holding all of its code: the producer / MMA warpgroup drops to
  // kRegsOther, the softmax warpgroups rise to kRegsSoftmax
  // (2*128*kRegsSoftmax + 128*kRegsOther <= 384*168).
  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther) : "memory");
  if (warp == kWarpLoad) {
    // ============================================================ TMA producer
    // The whole warp runs the loop (every branch below is warp-uniform); one
    // elected lane issues each copy and byte-count arrival.
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
    }
    __syncwarp();
    int u = 0;  // ring tiles loaded
    int g = 0;  // Q tiles loaded
    bool ok = true;
    // Q tile i of the item into slot g % 3, once the slot's previous tile is
    // done with.
    auto load_q = [&](const Work& w, int i) -> bool {
      const int slot = g % kQSlots, use = g / kQSlots;
      if (use > 0 &&
          !mbar_wait_warp(&q_empty[slot], (use - 1) & 1, abort_flag, p.wait_limit_ns))
        return false;
      mbar_arrive_expect_tx_w(&q_full[slot], C::kTileBytes);
#pragma unroll
      for (int a = 0; a < C::kAtoms; ++a)
        tma_load_4d_w(sQ + slot * C::kTileBytes + a * C::kAtomBytes, &tmQ, &q_full[slot], a * 64,
                      w.h, w.q_base + w.q0 + i * kBM, w.b_coord);
      ++g;
      return true;
    };
    // Key or value tile j of the item into one ring slot (its barrier's
    // byte count is one whole tile).  Dense and packed layouts: one box of
    // 128 rows per swizzle atom.  Paged cache: one 16-row box per page, lane
    // pp holding the page of rows 16pp.. (pages past the sequence's last are
    // replaced by that last page, whose rows are masked), read from the page
    // table one tile ahead of the loads and shared by the tile's K and V:
    // looked up twice per tile, just before each load, the chunked-prefill
    // workload took 0.387 ms against 0.349.  A page index outside the pool
    // is reported and page 0 read instead.
    auto lookup = [&](const Work& w, int j) -> int {
      int phys = 0;
      if (lane < kPagesPerTile) {
        const int np = (w.Lk + kPage - 1) / kPage;
        const int lp = min(j * kPagesPerTile + lane, np - 1);
        phys = p.page_table[static_cast<size_t>(w.bseq) * p.max_pages + lp];
      }
      return phys;
    };
    auto load_kv = [&](const CUtensorMap* map, uint8_t* dst, uint64_t* bar, const Work& w, int j,
                       int phys) {
      if constexpr (!kPagedKV) {
        (void)phys;
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a)
          tma_load_4d_w(dst + a * C::kAtomBytes, map, bar, a * 64, w.hk, w.k_base + j * kBN,
                        w.b_coord);
        return;
      } else {
        // lane pp issues the boxes of its own page: one warp instruction
        // starts the copies of all eight pages of an atom
        if (lane < kPagesPerTile) {
#pragma unroll
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_4d(dst + a * C::kAtomBytes + lane * kPage * 128, map, bar, a * 64, w.hk, 0,
                        phys);
        }
        __syncwarp();
      }
    };
    for (int c = 0; ok; ++c) {
      Work w;
      {
        if (!take_item(c)) {
          ok = false;
          break;
        }
        const ItemRec& r = recs[c % kRecSlots];
        if (!r.live) break;
        w = r.w;
        release_item(c);
      }
      if (w.lastT < 0) continue;
      if (!load_q(w, 0)) {
        ok = false;
        break;
      }
      // Warm L2 with the next item's Q tiles, if its record is out already.
      if (__all_sync(0xffffffffu, mbar_test(&rec_full[(c + 1) % kRecSlots],
                                            ((c + 1) / kRecSlots) & 1))) {
        const ItemRec& r2 = recs[(c + 1) % kRecSlots];
        if (r2.live && r2.w.lastT >= 0) {
#pragma unroll
          for (int i = 0; i < kQT; ++i)
#pragma unroll
            for (int a = 0; a < C::kAtoms; ++a)
              tma_prefetch_4d_w(&tmQ, a * 64, r2.w.h, r2.w.q_base + r2.w.q0 + i * kBM,
                                r2.w.b_coord);
        }
      }
      bool q1 = false;  // Q tile 1 loaded (after the item's first K tile)
      int phys = 0;  // paged cache: this lane's page of the current tile
      if constexpr (kPagedKV) phys = lookup(w, next_in_pair(w.r0, w.r1, 0, sinkT));
      for (int j = next_in_pair(w.r0, w.r1, 0, sinkT); j <= w.lastT;
           j = next_in_pair(w.r0, w.r1, j + 1, sinkT)) {
        const int s = u % ST;
        int phys_next = 0;
        if constexpr (kPagedKV) {
          // the next tile's pages in flight while this one is issued; an
          // index outside the pool is reported and page 0 read instead
          const int jn = next_in_pair(w.r0, w.r1, j + 1, sinkT);
          if (jn <= w.lastT) phys_next = lookup(w, jn);
          if (lane < kPagesPerTile && (phys < 0 || phys >= p.num_pages)) {
            atomicOr(p.status, kStatusBadInput);
            phys = 0;
          }
        }
        if (u >= ST &&
            !mbar_wait_warp(&step[s], ((u / ST) - 1) & 1, abort_flag, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        // Warm L2 with the key and value tiles kPrefetch active tiles ahead:
        // a ring slot is refilled only about one key step before it is read,
        // less than a load from HBM takes.
        {
          int jp = j, ahead = 0;
          while (ahead < kPrefetch) {
            const int nx = next_in_pair(w.r0, w.r1, jp + 1, sinkT);
            if (nx > w.lastT) break;
            jp = nx;
            ++ahead;
          }
          if (ahead == kPrefetch && !kPagedKV) {
#pragma unroll
            for (int a = 0; a < C::kAtoms; ++a) {
              tma_prefetch_4d_w(&tmK, a * 64, w.hk, w.k_base + jp * kBN, w.b_coord);
              tma_prefetch_4d_w(&tmV, a * 64, w.hk, w.k_base + jp * kBN, w.b_coord);
            }
          }
        }
        mbar_arrive_expect_tx_w(&k_full[s], C::kTileBytes);
        load_kv(&tmK, sK + s * C::kTileBytes, &k_full[s], w, j, phys);
        if (!q1) {
          // Between the first K and V tiles: S_0 of the first key step needs
          // K, S_1 needs this tile, and the first P V needs V last.
          q1 = true;
          if (!load_q(w, 1)) {
            ok = false;
            break;
          }
        }
        if (u >= ST && !mbar_wait_warp(&step[(u + 1) % ST], (((u + 1) / ST) - 1) & 1, abort_flag,
                                       p.wait_limit_ns)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx_w(&v_full[s], C::kTileBytes);
        load_kv(&tmV, sV + s * C::kTileBytes, &v_full[s], w, j, phys);
        phys = phys_next;
        ++u;
      }
      if (ok && !q1 && !load_q(w, 1)) ok = false;
    }
    // Tail: the last commit of the MMA issuer is step u (the final products
    // P V); once it is done no tensor-core commit is left to arrive on this
    // CTA's barriers.
    if (ok && u > 0 &&
        !mbar_wait_warp(&step[u % ST], (u / ST) & 1, abort_flag, p.wait_limit_ns))
      ok = false;
    if (!ok && lane == 0) fail(p.status, abort_flag);
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ============================================================ MMA issuer
    // The whole warp runs the loop (warp-uniform control flow); one elected
    // lane issues every MMA and commit.  The tensor pipe queues only a few
    // MMAs, so the issuer's own latency between groups (barrier tests of the
    // order of 100 cycles each, commits) can leave it idle: the barriers a
    // group needs are tested together, and key step u ends with one commit
    // that releases both K(u) and V(u - 1).
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, kBN, false);
    constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, true);
    // Descriptors are built once; every operand of every MMA is a base
    // descriptor plus a compile-time offset in its 16-byte address field
    // (shared-memory offsets stay below 256 KB, so the field never carries).
    constexpr uint64_t kTileDesc = C::kTileBytes >> 4;
    const uint64_t dq0 = sdesc_sw128(smem_addr(sQ), 16, 1024);
    const uint64_t dk0 = sdesc_sw128(smem_addr(sK), 16, 1024);
    const uint64_t dv0 = sdesc_sw128(smem_addr(sV), C::kAtomBytes, 1024);
    int u = 0;             // key steps (ring tiles) issued
    int g = 0;             // Q tiles consumed
    int pv0 = 0, pv1 = 0;  // products P V issued per Q tile (p_half / p_ready phases)
    // The product O_i += P_i V still to be issued: its ring tile (-1: none),
    // whether it is the first of its item (it overwrites O) and the last (its
    // completion is the item's o_done).
    int pend0 = -1, pend1 = -1;
    bool first0 = false, first1 = false, last0 = false, last1 = false;
    bool ok = true;
    // O_i += P_i V for ring tile pend (its V and the p_half arrival of its P
    // already waited for): the first half of P (keys 0..63) right away, the
    // second half once the softmax has published it (p_ready).
    auto issue_pv = [&](int i, int& pend, int& pv, bool first, bool last) -> bool {
      const uint64_t dv = dv0 + static_cast<uint64_t>(pend % ST) * kTileDesc;
      const uint32_t tO = tmem + C::kColO + i * D;
      const uint32_t tP = tmem + i * kBN;
      mma_ts_k64_w(tO, tP, dv, idesc_o, first ? 0u : 1u);
      if (!mbar_wait_warp(&p_ready[i], pv & 1, abort_flag, p.wait_limit_ns)) return false;
      tc_fence_after_sync();
      mma_ts_k64_w(tO, tP + 32, dv + 4 * (2048 >> 4), idesc_o, 1u);
      ++pv;
      if (last) mma_commit_w(&o_done[i]);
      pend = -1;
      return true;
    };
    // S_i = Q_i K^T for the key tile with descriptor dk, Q_i in slot qs.
    auto issue_s = [&](int i, uint64_t dk, int qs) {
      const uint64_t dq = dq0 + static_cast<uint64_t>(qs) * kTileDesc;
      const uint32_t tS = tmem + i * kBN;
      if constexpr (D == 128)
        mma_ss_k128_w<(C::kAtomBytes >> 4)>(tS, dq, dk, idesc_s);
      else
        mma_ss_k64_w(tS, dq, dk, idesc_s);
      mma_commit_w(&s_full[i]);
    };
    for (int c = 0; ok; ++c) {
      Work w;
      int count0, count1;
      {
        if (!take_item(c)) {
          ok = false;
          break;
        }
        const ItemRec& r = recs[c % kRecSlots];
        if (!r.live) break;
        w = r.w;
        count0 = r.count0;
        count1 = r.count1;
        release_item(c);
      }
      if (w.lastT < 0) continue;
      const int qs0 = g % kQSlots, qs1 = (g + 1) % kQSlots;
      const uint32_t qp0 = (g / kQSlots) & 1, qp1 = ((g + 1) / kQSlots) & 1;
      g += kQT;
      int left0 = count0, left1 = count1;
      for (int j = next_in_pair(w.r0, w.r1, 0, sinkT); j <= w.lastT;
           j = next_in_pair(w.r0, w.r1, j + 1, sinkT)) {
        const bool a0 = in_range(w.r0, j, sinkT), a1 = in_range(w.r1, j, sinkT);
        const int s = u % ST;
        const int sv = (u + ST - 1) % ST;  // V(u - 1)
        const uint32_t pk = (u / ST) & 1, pvv = ((u - 1) / ST) & 1;
        // Needed now: K(u), and for O_0 += P_0 V(u - 1) also V(u - 1) and
        // the first half of P_0.  Tested together (one round trip when all
        // are ready), then waited on in turn only if one is not.  A barrier
        // not needed is replaced by K(u)'s own.
        const bool need_v = pend0 >= 0 || pend1 >= 0, need_p0 = pend0 >= 0;
        if (!__all_sync(0xffffffffu,
                        mbar_test3(&k_full[s], pk, need_v ? &v_full[sv] : &k_full[s],
                                   need_v ? pvv : pk, need_p0 ? &p_half[0] : &k_full[s],
                                   need_p0 ? (pv0 & 1) : pk) == 7u)) {
          if (!mbar_wait_warp(&k_full[s], pk, abort_flag, p.wait_limit_ns) ||
              (need_v && !mbar_wait_warp(&v_full[sv], pvv, abort_flag, p.wait_limit_ns)) ||
              (need_p0 && !mbar_wait_warp(&p_half[0], pv0 & 1, abort_flag, p.wait_limit_ns))) {
            ok = false;
            break;
          }
        }
        tc_fence_after_sync();
        const uint64_t dk = dk0 + static_cast<uint64_t>(s) * kTileDesc;
        // order: O_0 += P_0 V(u-1), S_0(u), O_1 += P_1 V(u-1), S_1(u)
        if (pend0 >= 0 && !issue_pv(0, pend0, pv0, first0, last0)) {
          ok = false;
          break;
        }
        if (a0) {
          // the item's first S_0 waits for its Q tile
          if (left0 == count0) {
            if (!mbar_wait_warp(&q_full[qs0], qp0, abort_flag, p.wait_limit_ns)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
          }
          issue_s(0, dk, qs0);
          first0 = left0 == count0;
          last0 = --left0 == 0;
          if (last0) mma_commit_w(&q_empty[qs0]);
          pend0 = u;
        }
        if (pend1 >= 0) {
          if (!mbar_wait_warp(&p_half[1], pv1 & 1, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          if (!issue_pv(1, pend1, pv1, first1, last1)) {
            ok = false;
            break;
          }
        }
        if (a1) {
          if (left1 == count1) {
            if (!mbar_wait_warp(&q_full[qs1], qp1, abort_flag, p.wait_limit_ns)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
          }
          issue_s(1, dk, qs1);
          first1 = left1 == count1;
          last1 = --left1 == 0;
          if (last1) mma_commit_w(&q_empty[qs1]);
          pend1 = u;
        }
        mma_commit_w(&step[s]);  // key step u: K(u) and V(u - 1) free once done
        ++u;
      }
      if (!ok) break;
      // A Q tile with no key tile to see: nothing reads it; hand its slot
      // back once it has landed.
      if (count0 == 0) {
        if (!mbar_wait_warp(&q_full[qs0], qp0, abort_flag, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        mma_commit_w(&q_empty[qs0]);
      }
      if (count1 == 0) {
        if (!mbar_wait_warp(&q_full[qs1], qp1, abort_flag, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        mma_commit_w(&q_empty[qs1]);
      }
    }
    // Final key step: the products of the last tile.
    if (ok && (pend0 >= 0 || pend1 >= 0)) {
      ok = mbar_wait_warp(&v_full[(u + ST - 1) % ST], ((u - 1) / ST) & 1, abort_flag,
                          p.wait_limit_ns);
      if (ok && pend0 >= 0) {
        ok = mbar_wait_warp(&p_half[0], pv0 & 1, abort_flag, p.wait_limit_ns);
        if (ok) {
          tc_fence_after_sync();
          ok = issue_pv(0, pend0, pv0, first0, last0);
        }
      }
      if (ok && pend1 >= 0) {
        ok = mbar_wait_warp(&p_half[1], pv1 & 1, abort_flag, p.wait_limit_ns);
        if (ok) {
          tc_fence_after_sync();
          ok = issue_pv(1, pend1, pv1, first1, last1);
        }
      }
      if (ok) mma_commit_w(&step[u % ST]);
    }
    if (!ok && lane == 0) fail(p.status, abort_flag);
    __syncwarp();
  } else if (warp == kWarpTable) {
    // ============================================================ item locator
    // Walks this CTA's items ahead of the other roles: one record per item
    // with query rows (items with invalid sequence offsets are reported here
    // and left out), then one with live = 0.  A slot is rewritten once all
    // kRecReaders warps have freed it, so the locator runs up to kRecSlots
    // items ahead of the slowest role and its table search and offset loads
    // stay off their item changes.
    bool ok = true;
    int c = 0;
    for (int n = 0; ok; ++n) {
      const int k = item_of(n, num_items);
      ItemLoc loc = {0, 0, 0, 0, 0, 0, 0};
      if (k >= 0 && !locate_item<kPagedKV, kTable>(p, tab, k, loc, lane == 0)) continue;
      ItemRec r;
      work_of<kPagedKV>(p, loc, r.w);
      r.count0 = range_count(r.w.r0, sinkT);
      r.count1 = range_count(r.w.r1, sinkT);
      r.live = k >= 0;
      const int rs = c % kRecSlots;
      if (c >= kRecSlots &&
          !mbar_wait_warp(&rec_empty[rs], ((c / kRecSlots) - 1) & 1, abort_flag, p.wait_limit_ns)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        recs[rs] = r;
        mbar_arrive(&rec_full[rs]);
      }
      __syncwarp();
      ++c;
      if (k < 0) break;
    }
    if (!ok && lane == 0) fail(p.status, abort_flag);
    __syncwarp();
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax) : "memory");
    // ============================================================ softmax warpgroups
    const int i = warp / 4;
    const int wq = warp % 4;
    const int r = wq * 32 + lane;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t colS = i * kBN;
    const uint32_t colO = C::kColO + i * D;
    const float scale2 = p.scale2;
    int t = 0;     // key tiles processed (s_full / p_ready phases)
    int no = 0;    // o_done phases consumed
    bool ok = true;
    for (int c = 0; ok; ++c) {
      // Only what the key loop needs stays live through it; the epilogue
      // reads the item's record again (this warp frees it after that).
      TileMask m;
      TileRange rg;
      int hi_row, lo_row;
      {
        if (!take_item(c)) {
          if (lane == 0) fail(p.status, abort_flag);
          ok = false;
          break;
        }
        const ItemRec& rec = recs[c % kRecSlots];
        if (!rec.live) break;
        const Work& w = rec.w;
        const int row = w.q0 + i * kBM + r;  // sequence-relative query index
        hi_row = p.causal ? min(row + w.off, w.Lk - 1) : w.Lk - 1;
        lo_row = (p.window > 0) ? row + w.off - p.window : kNoLowerBound;
        m = i ? w.m1 : w.m0;
        rg = i ? w.r1 : w.r0;
      }

      float m_used = -INFINITY;  // raw (unscaled) running maximum in use
      float l = 0.f;             // running sum of the fp32 probabilities
      float corr = 0.f;          // running sum of (p - bf16(p)) over each tile's largest p
      int t_item = 0;
      for (int j = next_in_range(rg, 0, sinkT); j <= rg.hi; j = next_in_range(rg, j + 1, sinkT)) {
        bool w_ok = mbar_wait(&s_full[i], t & 1, abort_flag, p.wait_limit_ns);
        w_ok = __all_sync(0xffffffffu, w_ok);
        if (!w_ok) {
          if (lane == 0) fail(p.status, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const bool edge = !tile_interior(m, j, p.window, p.n_sink);
        const uint32_t sS = taddr + colS;
        uint64_t sum_a = 0, sum_b = 0;  // bit pattern 0 is (+0.f, +0.f)
        float mx = -INFINITY;
        bool do_rescale = false;
        float alpha = 1.f;
        float ms = 0.f;
        // P goes over the first 64 columns of S as bf16 pairs: the P of score
        // chunk c (32 columns) to columns 16c..16c+15, on scores already read.
        // P of keys 0..63 is published (p_half) as soon as it is written, so
        // the tensor core starts the second product on it while keys 64..127
        // are still exponentiated; p_ready follows the rest.
        //
        // Interior tile after the first of the item: speculate that no row's
        // maximum grows past the rescale threshold, so the maximum in use
        // stays.  Chunks 0 and 1 are exponentiated with it as they arrive,
        // chunks 2 and 3 are held; once the whole tile's maximum confirms the
        // guess, the first half of P is written and published and the second
        // half formed.  If a row of the warp does exceed the threshold (rare
        // after the first tile), nothing has been written yet: the warp
        // starts again on the full path below, S being intact.
        //
        // The first tile of an item (no maximum in use yet) is speculated
        // the same way, with the maximum of its first chunk as the guess.
        bool spec_ok = false;
        if (!edge) {
          const bool first = m_used == -INFINITY;  // uniform: every row starts the item together
          uint32_t ra[32], rb[32], pk0[16], pk1[16];
          tmem_ld_x32(sS + 0, ra);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) reg_fence(ra[c]);
          tmem_ld_x32(sS + 32, rb);
          float mxa = max32(ra, -INFINITY);
          if (first) m_used = mxa;
          ms = m_used * scale2;
          const uint64_t sc2 = f2(scale2, scale2), nms = f2(-ms, -ms);
          exp32(ra, sc2, nms, sum_a, sum_b, pk0);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) reg_fence(rb[c]);
          tmem_ld_x32(sS + 64, ra);
          mxa = max32(rb, mxa);
          exp32(rb, sc2, nms, sum_a, sum_b, pk1);
          tmem_ld_x32(sS + 96, rb);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            reg_fence(ra[c]);
            reg_fence(rb[c]);
          }
          mx = max32(rb, max32(ra, mxa));
          if (!__any_sync(0xffffffffu, (mx - m_used) * scale2 > kRescaleLog2)) {
            tmem_st_x16(sS + 0, pk0);
            tmem_st_x16(sS + 16, pk1);
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&p_half[i]);
            exp32(ra, sc2, nms, sum_a, sum_b, pk0);
            tmem_st_x16(sS + 32, pk0);
            exp32(rb, sc2, nms, sum_a, sum_b, pk1);
            tmem_st_x16(sS + 48, pk1);
            spec_ok = true;
          } else {
            sum_a = sum_b = 0;  // start again
            mx = -INFINITY;
            if (first) m_used = -INFINITY;
          }
        }
        // Online-softmax state update from this tile's raw row maximum, and
        // the rescale of O it may need.  O of this row was last written by the
        // product issued before S(j), which has completed (the commit behind
        // s_full covers it); the next product into O waits for the p_half
        // arrival that follows, so the rescale comes before any P is
        // published.
        auto update_rescale = [&]() {
          if (mx > m_used) {
            if (m_used == -INFINITY) {
              m_used = mx;
            } else if ((mx - m_used) * scale2 > kRescaleLog2) {
              alpha = ex2_approx((m_used - mx) * scale2);
              l *= alpha;
              corr *= alpha;
              m_used = mx;
              do_rescale = true;
            }
          }
          ms = (m_used == -INFINITY) ? 0.f : m_used * scale2;
          if (__any_sync(0xffffffffu, do_rescale)) {
            const uint64_t a2 = f2(alpha, alpha);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t ro[32];
              tmem_ld_x32(taddr + colO + c * 32, ro);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                reg_fence(ro[2 * e]);
                reg_fence(ro[2 * e + 1]);
                float o0, o1;
                f2_split(f2_mul(f2(__uint_as_float(ro[2 * e]), __uint_as_float(ro[2 * e + 1])), a2),
                         o0, o1);
                ro[2 * e] = __float_as_uint(o0);
                ro[2 * e + 1] = __float_as_uint(o1);
              }
              tmem_st_x32(taddr + colO + c * 32, ro);
            }
          }
        };
        if (spec_ok) {
        } else {
          // First tile of the item, or a tile a boundary crosses (causal
          // diagonal, window edge, sink keys, ragged tail): all of S in
          // registers (one wait), the mask on boundary tiles, the row maximum
          // and the state update, then the exponentials from the registers,
          // publishing the first half of P once chunks 0 and 1 are written.
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tmem_ld_x32(sS + 0, r0);
          tmem_ld_x32(sS + 32, r1);
          tmem_ld_x32(sS + 64, r2);
          tmem_ld_x32(sS + 96, r3);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            reg_fence(r0[c]);
            reg_fence(r1[c]);
            reg_fence(r2[c]);
            reg_fence(r3[c]);
          }
          if (edge) {
            const int kb = j * kBN;
            const int lim_hi = hi_row - kb;
            const int lim_lo = (p.window > 0) ? lo_row - kb : kNoLowerBound;
            const int lim_sink = p.n_sink - kb;
            mask32(r0, lim_hi, lim_lo, lim_sink);
            mask32(r1, lim_hi - 32, lim_lo - 32, lim_sink - 32);
            mask32(r2, lim_hi - 64, lim_lo - 64, lim_sink - 64);
            mask32(r3, lim_hi - 96, lim_lo - 96, lim_sink - 96);
          }
          mx = max32(r3, max32(r2, max32(r1, max32(r0, mx))));
          update_rescale();
          const uint64_t sc2 = f2(scale2, scale2), nms = f2(-ms, -ms);
          uint32_t pk[16];
          exp32(r0, sc2, nms, sum_a, sum_b, pk);
          tmem_st_x16(sS + 0, pk);
          exp32(r1, sc2, nms, sum_a, sum_b, pk);
          tmem_st_x16(sS + 16, pk);
          tmem_st_wait();
          tc_fence_before_sync();
          mbar_arrive(&p_half[i]);
          exp32(r2, sc2, nms, sum_a, sum_b, pk);
          tmem_st_x16(sS + 32, pk);
          exp32(r3, sc2, nms, sum_a, sum_b, pk);
          tmem_st_x16(sS + 48, pk);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&p_ready[i]);
        float s0, s1, s2, s3;
        f2_split(sum_a, s0, s1);
        f2_split(sum_b, s2, s3);
        l += (s0 + s1) + (s2 + s3);
        // The second product sees bf16-rounded probabilities.  When one key
        // dominates a row, its rounding error would not cancel between O and
        // l; track it for the largest probability of every tile (recomputed
        // with the arithmetic exp32 used for it, so the same value) and take
        // it out of the normaliser of O.
        {
          const float ptop = ex2_approx(__fmaf_rn(mx, scale2, -ms));
          const float ptop_r = __uint_as_float(pack_bf16x2(0.f, ptop) & 0xffff0000u);
          corr += ptop - ptop_r;
        }
        ++t;
        ++t_item;
      }
      if (!ok) break;

      // ---------------------------------------------------------------- epilogue
      // O / l in bf16 straight from tensor memory to the caller's layout
      // (each thread its own row, 16-byte stores), then the row's LSE.  Every
      // branch below is uniform over the warp, and the tensor-memory loads
      // (warp-collective) are made by every lane whatever its row.
      const Work& w = recs[c % kRecSlots].w;
      const int row = w.q0 + i * kBM + r;
      const bool valid = row < w.Lq;
      const bool have_o = t_item > 0;
      if (have_o) {
        bool w_ok = mbar_wait(&o_done[i], no & 1, abort_flag, p.wait_limit_ns);
        w_ok = __all_sync(0xffffffffu, w_ok);
        ++no;
        if (!w_ok) {
          if (lane == 0) fail(p.status, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after_sync();
      }
      const bool seen = have_o && l > 0.f;
      // Logit sink sigma of this head ("TileLang tutorial, ch.15", section
      // 4.6): one more term of the denominator, taken against
      // m* = max(sigma, m * scale) so that it cannot overflow; with no sink
      // (-inf) the plain normalisation.
      const float sg = p.sink ? p.sink[w.h] : -INFINITY;
      float inv, lse_row;
      if (sg == -INFINITY) {
        inv = seen ? 1.f / (l - corr) : 0.f;
        lse_row = seen ? fmaf(m_used, p.scale, logf(l)) : -INFINITY;
      } else {
        const float a = seen ? m_used * p.scale : -INFINITY;
        const float mst = fmaxf(a, sg);
        const float e1 = seen ? expf(a - mst) : 0.f;
        const float e2 = expf(sg - mst);
        inv = e1 / fmaf(l - corr, e1, e2);
        lse_row = mst + logf(fmaf(l, e1, e2));
      }
      {
        const uint64_t inv2 = f2(inv, inv);
        uint4* dst = reinterpret_cast<uint4*>(
            p.o + static_cast<long long>(w.bseq) * p.o_sb +
            static_cast<long long>(w.q_base + row) * p.o_ss + static_cast<long long>(w.h) * p.o_sh);
        // 32 columns at a time, the next chunk's load in flight while one is
        // scaled, packed and stored.
        // Each thread stores its own row, so one store instruction touches
        // 32 rows; 32-byte stores halve the instructions (and the requests
        // the L1 processes) against 16-byte ones.
        auto store32 = [&](const uint32_t* o, int c) {
          uint32_t wv[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float a0, a1;
            f2_split(f2_mul(f2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), inv2), a0,
                     a1);
            wv[e] = seen ? pack_bf16x2(a0, a1) : 0u;
          }
          if (valid) {
            if (p.o_v8) {
              st_global_v8(dst + c * 4, wv);
              st_global_v8(dst + c * 4 + 2, wv + 8);
            } else {
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4)
                dst[c * 4 + v4] = make_uint4(wv[4 * v4], wv[4 * v4 + 1], wv[4 * v4 + 2], wv[4 * v4 + 3]);
            }
          }
        };
        uint32_t oa[32], ob[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) oa[e] = ob[e] = 0u;
        if (have_o) {
          tmem_ld_x32(taddr + colO, oa);
          tmem_ld_wait();
        }
        // Not unrolled: the epilogue runs once per item, and as straight-line
        // code it missed the instruction cache chunk after chunk (measured:
        // rolled, the window call 102.7 -> 100.4 us, GQA causal 194.5 -> 192.0).
#pragma unroll 1
        for (int c = 0; c < D / 32; c += 2) {
#pragma unroll
          for (int e = 0; e < 32; ++e) reg_fence(oa[e]);
          if (have_o) tmem_ld_x32(taddr + colO + (c + 1) * 32, ob);
          store32(oa, c);
          if (have_o) tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) reg_fence(ob[e]);
          if (have_o && c + 2 < D / 32) tmem_ld_x32(taddr + colO + (c + 2) * 32, oa);
          store32(ob, c + 1);
          if (have_o && c + 2 < D / 32) tmem_ld_wait();
        }
      }
      if (valid && p.lse != nullptr) {
        const size_t li = p.cu_q ? static_cast<size_t>(w.h) * p.total_q + w.q_base + row
                                 : (static_cast<size_t>(w.bseq) * p.Hq + w.h) * p.Sq + row;
        p.lse[li] = lse_row;
      }
      // The next item's first product into O must wait until O has been read:
      // it waits for this warpgroup's next p_half arrival, made after this.
      tc_fence_before_sync();
      release_item(c);
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before_sync();
  __syncthreads();
  if (*abort_flag) {
    // Let every tensor-core operation and bulk copy already issued land
    // before the tensor memory and shared memory are given back.
    if (warp == kWarpMma) {
      mma_commit_w(drain);
      mbar_wait_warp(drain, 0, nullptr, 100000000ull);
    }
    if (warp == kWarpLoad && lane == 0) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) {
      }
    }
    __syncthreads();
  }
  tc_fence_after_sync();
  if (warp == kWarpLoad) tmem_dealloc(tmem, C::kTmemCols);
}

// O = 0 and LSE = -inf (or the head's logit sink) everywhere: every query
// sees no key (no keys at all).  LSE element e belongs to head
// (e / lse_inner) % Hq.
// O element e of row r = b * lse_inner + s, head h, column t lives at
// b * sb + s * ss + h * sh + t (the caller's strides, in elements).
__global__ void attn_fill_empty_kernel(__nv_bfloat16* o, size_t o_elems, float* lse,
                                       size_t lse_elems, const float* sink, size_t lse_inner,
                                       int Hq, int d, long long sb, long long ss, long long sh) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t e = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; e < o_elems;
       e += stride) {
    const size_t t = e % static_cast<size_t>(d), hr = e / static_cast<size_t>(d);
    const size_t h = hr % static_cast<size_t>(Hq), r = hr / static_cast<size_t>(Hq);
    const size_t b = r / lse_inner, sq = r % lse_inner;
    o[b * sb + sq * ss + h * sh + t] = __float2bfloat16(0.f);
  }
  if (lse)
    for (size_t e = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; e < lse_elems;
         e += stride)
      lse[e] = sink ? sink[(e / lse_inner) % static_cast<size_t>(Hq)] : -INFINITY;
}

template <int D>
cudaError_t launch_d(const FwdLaunch& a, cudaStream_t stream) {
  using C = Cfg<D>;
  // dynamic shared memory plus the static table, item records and flags
  // within the 227 KB a block may have
  static_assert(C::kSmemBytes + sizeof(ItemTable) + kRecSlots * sizeof(ItemRec) + 64 <=
                    227 * 1024,
                "shared memory");
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    for (auto fn : {attn_fwd_kernel<D, false, false>, attn_fwd_kernel<D, true, false>,
                    attn_fwd_kernel<D, false, true>, attn_fwd_kernel<D, true, true>}) {
      attr_err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      C::kSmemBytes);
      if (attr_err != cudaSuccess) return;
      // setmaxnreg.inc waits for registers the block was launched with:
      // never launch a build whose register count cannot cover the split.
      cudaFuncAttributes fa;
      attr_err = cudaFuncGetAttributes(&fa, fn);
      if (attr_err == cudaSuccess && fa.numRegs * kThreads < kRegsSplit)
        attr_err = cudaErrorInvalidConfiguration;
      if (attr_err != cudaSuccess) return;
    }
  });
  if (attr_err != cudaSuccess) return attr_err;
  Params p;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.o_sb = a.o_sb;
  p.o_ss = a.o_ss;
  p.o_sh = a.o_sh;
  p.o_v8 = (reinterpret_cast<uintptr_t>(a.o) % 32 == 0) && a.o_sb % 16 == 0 && a.o_ss % 16 == 0 &&
           a.o_sh % 16 == 0;
  p.lse = a.lse;
  p.sink = a.sink;
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.page_table = a.page_table;
  p.seqlens_k = a.seqlens_k;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Skv = a.Skv;
  p.total_q = a.total_q;
  p.num_qpairs = (a.Sq + kQT * kBM - 1) / (kQT * kBM);
  p.div_hq = make_fastdiv(static_cast<uint32_t>(a.Hq));
  p.div_b = make_fastdiv(static_cast<uint32_t>(std::max(a.B, 1)));
  p.div_qp = make_fastdiv(static_cast<uint32_t>(std::max(p.num_qpairs, 1)));
  p.div_group = make_fastdiv(static_cast<uint32_t>(a.Hq / a.Hkv));
  p.scale = a.scale;
  p.scale2 = a.scale * kLog2e;
  p.causal = a.causal;
  p.window = a.window;
  p.n_sink = a.n_sink;
  p.wait_limit_ns = kWaitLimitNs;
  p.status = a.status;
  const long long items = static_cast<long long>(p.num_qpairs) * a.B * a.Hq;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  p.num_items = static_cast<int>(items);
  // Persistent: one CTA per SM (shared and tensor memory hold one), each
  // walking its share of the items.
  const int grid = static_cast<int>(std::min<long long>(items, std::max(a.num_sms, 1)));
  // The paged cache has an instantiation of its own, so that the dense and
  // packed kernels' code is not touched by its page lookups.
  // Causal packed calls small enough for the dense item order get the
  // instantiation that builds and walks it.
  const bool table = a.cu_q != nullptr && a.causal && a.B <= kTabMaxSeq &&
                     p.num_qpairs <= kTabMaxLev;
  if (a.page_table != nullptr) {
    if (table)
      attn_fwd_kernel<D, true, true><<<grid, kThreads, C::kSmemBytes, stream>>>(a.tmQ, a.tmK,
                                                                              a.tmV, p);
    else
      attn_fwd_kernel<D, true, false><<<grid, kThreads, C::kSmemBytes, stream>>>(a.tmQ, a.tmK,
                                                                               a.tmV, p);
  } else if (table) {
    attn_fwd_kernel<D, false, true><<<grid, kThreads, C::kSmemBytes, stream>>>(a.tmQ, a.tmK,
                                                                             a.tmV, p);
  } else {
    attn_fwd_kernel<D, false, false><<<grid, kThreads, C::kSmemBytes, stream>>>(a.tmQ, a.tmK,
                                                                              a.tmV, p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const FwdLaunch& a, cudaStream_t stream) {
  if (a.d == 128) return launch_d<128>(a, stream);
  if (a.d == 64) return launch_d<64>(a, stream);
  if (a.d == 256) return launch_attn_fwd256(a, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_fill_empty(const FwdLaunch& a, cudaStream_t stream) {
  const size_t rows = a.cu_q ? static_cast<size_t>(a.total_q) : static_cast<size_t>(a.B) * a.Sq;
  const size_t o_elems = rows * a.Hq * a.d;
  const size_t lse_elems = rows * a.Hq;
  if (o_elems == 0) return cudaSuccess;
  const size_t lse_inner = a.cu_q ? static_cast<size_t>(a.total_q) : static_cast<size_t>(a.Sq);
  attn_fill_empty_kernel<<<1216, 256, 0, stream>>>(static_cast<__nv_bfloat16*>(a.o), o_elems,
                                                   a.lse, lse_elems, a.sink, lse_inner, a.Hq, a.d,
                                                   a.o_sb, a.o_ss, a.o_sh);
  return cudaGetLastError();
}

}  // namespace attn
