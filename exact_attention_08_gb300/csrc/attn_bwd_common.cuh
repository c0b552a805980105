// Shared pieces of the backward kernels (d = 64 / 128 in attn_bwd_sm103.cu,
// d = 256 in attn_bwd256_sm103.cu): the launch parameters, per-sequence
// geometry, packed-float helpers, bounded waits and row stores.
#pragma once

#include "attn_internal.h"
#include "sm103_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace attn {

struct BwdParams {
  const __nv_bfloat16* dout;  // [B, Sq, Hq, d] or packed [total_q, Hq, d] (row statistics only)
  const __nv_bfloat16* o;
  const __nv_bfloat16* v;     // [B, Skv, Hkv, d] or packed (d = 256: V rows into tensor memory)
  const float* lse;          // [B, Hq, Sq] or packed [Hq, total_q], natural log
  const int* cu_q;           // packed sequences: [B + 1] query offsets, or null (dense)
  const int* cu_k;           // packed sequences: [B + 1] key offsets
  float* lse2;               // [B, Hq, Sqp] workspace: -LSE * log2(e), -inf on pad rows
  float* dvec;               // [B, Hq, Sqp] workspace: -rowsum(dO * O)
  __nv_bfloat16* dq;         // [B, Sq, Hq, d]
  __nv_bfloat16* dk;         // [B, Skv, Hkv, d]
  __nv_bfloat16* dv;
  int v8;                    // dq, dk and dv start on 32 bytes: 32-byte stores
  int B, Hq, Hkv, Sq, Skv, Sqp, d;  // Sq, Skv: the longest sequence when packed
  int total_q, total_k;             // packed token counts
  float scale, scale2;
  int causal, window, n_sink;
  uint64_t wait_limit_ns;
  int* status;
};

// The d = 256 gradient kernels (dV, dK, then dQ, one launch each), launched
// after the row statistics of attn_bwd_sm103.cu have filled p.lse2 / p.dvec.
cudaError_t launch_bwd256(const BwdParams& p, const BwdLaunch& a, cudaStream_t stream);

namespace {

using namespace ptx;

constexpr int kB = 128;          // rows of every tile (keys or queries)
// Warps 0-7 compute, 8 producer, 9 MMA.  Compute warp w reads tensor-memory
// lanes 32 (w % 4) .. +31 (its sub-partition's quarter) and the column half
// w / 4 of every 128-column tile, so each sub-partition runs two of them.
constexpr int kComputeWarps = 8;
constexpr int kBwdThreads = 32 * (kComputeWarps + 2);
constexpr int kWarpProd = kComputeWarps;
constexpr int kWarpIssue = kComputeWarps + 1;
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr float kLog2eB = 1.4426950408889634f;

// One sequence's geometry: lengths, first rows in the tensors (for
// addressing outputs), and the TMA coordinates of its first rows.
struct SeqGeo {
  int Lq, Lk, q_base, k_base, b_coord;
  long long q_row0, k_row0;
};

// False (and reported when `report`) for packed offsets out of range.
__device__ __forceinline__ bool seq_geo(const BwdParams& p, int b, SeqGeo& g, bool report) {
  if (p.cu_q != nullptr) {
    const int a = p.cu_q[b], e = p.cu_q[b + 1], ka = p.cu_k[b], ke = p.cu_k[b + 1];
    if (a < 0 || e < a || e > p.total_q || e - a > p.Sq || ka < 0 || ke < ka ||
        ke > p.total_k || ke - ka > p.Skv) {
      if (report) atomicOr(p.status, kStatusBadInput);
      return false;
    }
    g.Lq = e - a;
    g.Lk = ke - ka;
    g.q_base = a;
    g.k_base = ka;
    g.b_coord = 0;
    g.q_row0 = a;
    g.k_row0 = ka;
  } else {
    g.Lq = p.Sq;
    g.Lk = p.Skv;
    g.q_base = 0;
    g.k_base = 0;
    g.b_coord = b;
    g.q_row0 = static_cast<long long>(b) * p.Sq;
    g.k_row0 = static_cast<long long>(b) * p.Skv;
  }
  return true;
}

__device__ __forceinline__ void reg_fence_b(uint32_t& r) { asm volatile("" : "+r"(r)); }

__device__ __forceinline__ uint64_t pf2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void pf2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t pf2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t pf2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t pf2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Four consecutive floats of shared memory as two pairs (one 16-byte load).
// Volatile, so it stays after the barrier wait that makes the data valid.
__device__ __forceinline__ void lds_pairs2(uint32_t addr, uint64_t& a, uint64_t& b) {
  asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(addr));
}
// One 32-column chunk of a row vector: 16 pairs.
__device__ __forceinline__ void lds_chunk(uint32_t addr, uint64_t* v) {
#pragma unroll
  for (int i = 0; i < 8; ++i) lds_pairs2(addr + 16 * i, v[2 * i], v[2 * i + 1]);
}

__device__ __forceinline__ void tmem_ld_wait_b() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// A 128-column fp32 tile rewritten in place as bf16 pairs: the 32-column
// chunk c goes to 16 columns at 64 (c / 2) + 16 (c % 2), inside the column
// half that holds its source, so the warp that reads a half is the only one
// that writes it.  K-step kk (16 columns of the tile) of an MMA that takes
// the packed tile as its A operand starts at packed_col(kk).
__device__ __forceinline__ uint32_t packed_col(int kk) {
  return static_cast<uint32_t>(64 * (kk / 4) + 8 * (kk % 4));
}

__device__ __forceinline__ void bwd_fail(int* status, volatile int* abort_flag) {
  atomicOr(status, kStatusTimeout);
  if (abort_flag) *abort_flag = 1;
}

// Packs 32 fp32 values into 16 bf16 pairs (element 2e in the low half).
__device__ __forceinline__ void pack32(const float* f, uint32_t* pk) {
#pragma unroll
  for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(f[2 * e], f[2 * e + 1]);
}

// 32 bf16 (16 pairs) of one row to global memory: two 32-byte stores when
// the row is 32-byte aligned (each thread stores its own row, so a store
// instruction touches 32 rows and fewer, wider ones cost the L1 less), else
// four 16-byte stores.
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t* pk, int v8) {
  if (v8) {
    st_global_v8(dst, pk);
    st_global_v8(dst + 16, pk + 8);
  } else {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int v4 = 0; v4 < 4; ++v4)
      d4[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
  }
}

// K-step kk of a K-major SW128 operand: 32 bytes along a row inside a
// 128-byte atom, then the next atom column.
template <int kAtomBytes>
__device__ __forceinline__ uint64_t kmajor_step(int kk) {
  return static_cast<uint64_t>(((kk / 4) * kAtomBytes + (kk % 4) * 32) >> 4);
}

// Bounded wait by every lane of the warp; on failure the status is set once.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          const BwdParams& p) {
  const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.wait_limit_ns));
  if (!ok && (threadIdx.x % 32) == 0) bwd_fail(p.status, abort_flag);
  return ok;
}

// The n-th item of this CTA, or -1 past the last: bands of gridDim.x items,
// every other band dealt in reverse CTA order.  With one CTA per item (the
// grid as large as the item count) every CTA takes its own item only.
__device__ __forceinline__ int bwd_item_at(int n, int num_items) {
  const int G = gridDim.x;
  const int pos = (n & 1) ? (G - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  const long long k = static_cast<long long>(n) * G + pos;
  return k < num_items ? static_cast<int>(k) : -1;
}

// The gradient kernels of one call form a programmatic launch chain.  They
// read the inputs and the row statistics, never one another's outputs, so a
// kernel may start on the SMs its predecessor frees.  Every CTA allows its
// dependents as it starts, and before it exits it waits for its
// predecessor's grid to complete, so that the last kernel's completion
// still implies every earlier one's.  In a kernel launched without the
// programmatic attribute both return at once.
__device__ __forceinline__ void chain_allow_next() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void chain_join_prev() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launch of a gradient kernel as the programmatic dependent of the kernel
// before it on the stream.
template <typename Kernel, typename... Args>
cudaError_t launch_chained(Kernel kernel, unsigned grid, size_t smem, cudaStream_t stream,
                           Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kBwdThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace
}  // namespace attn
