// Internal interface between the C-ABI host code and the kernel translation
// units.  Not installed; not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

// device status bits (the status word is an int in device memory)
enum : int {
  kStatusTimeout = 1,   // a bounded wait ran out
  kStatusBadInput = 2,  // out-of-range device data (page index, cu_seqlens)
  kStatusLayout = 4,    // a kernel's shared-memory window was not where its layout needs it
};

// Default limit of every bounded wait in the production kernels.
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s

struct FwdLaunch {
  CUtensorMap tmQ, tmK, tmV, tmO;  // 4-D maps (d, H, S, B) with 64 x 1 x 128 x 1 boxes
  void* o;                    // bf16 output
  float* lse;                 // fp32 log-sum-exp, may be null
  const float* sink;          // fp32 logit sink per query head [Hq], may be null
  const int* cu_q;            // null: dense layout
  const int* cu_k;
  const int* page_table;      // paged K/V [B, max_pages], or null
  const int* seqlens_k;       // paged K/V key counts [B]
  int max_pages, num_pages;
  long long o_sb, o_ss, o_sh;  // O strides (elements) of batch, row and head; d contiguous
  int B, Hq, Hkv;
  int Sq, Skv;                // dense sizes, or the maxima for varlen
  int total_q, total_k;       // varlen totals (dense: unused)
  int d;
  float scale;
  int causal, window, n_sink;
  int num_sms;  // SMs of the device (the persistent grid)
  int* status;
};

struct DecodeLaunch {
  CUtensorMap tmK, tmV;  // 4-D maps over the page pools (d, Hkv, page, pages), 64 x 1 x 16 x 1 boxes
  const void* q;
  void* o;
  float* lse;
  const float* sink;  // fp32 logit sink per query head [Hq], may be null
  const int* page_table;
  const int* seqlens;
  float* ws_o;    // [B, Hq, S, d] fp32 split outputs (normalised)
  float* ws_lse;  // [B, Hq, S] fp32 split log-sum-exps (natural log)
  int* order;     // [B] workspace: the requests longest first
  int B, Hq, Hkv, d, page, max_pages, num_pages, num_splits;
  float scale;
  int* status;
};

struct BwdLaunch {
  CUtensorMap tmQ, tmK, tmV, tmDO;  // 4-D maps (d, H, S, B), 64 x 1 x 128 x 1 boxes
                                    // (64 x 1 x 64 x 1 at d = 256)
  const void* v;                    // bf16 values [B, Skv, Hkv, d] or [total_k, Hkv, d]
  const void* o;                    // bf16 forward output [B, Sq, Hq, d] or [total_q, Hq, d]
  const void* dout;                 // bf16 gradient of O, same layout
  const float* lse;                 // forward LSE [B, Hq, Sq] or [Hq, total_q] (natural log)
  void* dq;                         // bf16, the layout of q
  void* dk;                         // bf16 [B, Skv, Hkv, d] or [total_k, Hkv, d]
  void* dv;
  float* ws_lse2;                   // [B, Hq, Sqp] fp32 workspace
  float* ws_d;                      // [B, Hq, Sqp] fp32 workspace
  const int* cu_q;                  // packed sequences: [B + 1] offsets, or null (dense)
  const int* cu_k;
  const float* sink;                // logit sink per query head [Hq], or null
  float* dsink;                     // its gradient [Hq] (written when sink is set)
  int total_q, total_k;             // packed token counts
  int B, Hq, Hkv, Sq, Skv, d;       // Sq, Skv: the longest sequence when packed
  float scale;
  int causal, window, n_sink;
  int* status;
  int num_sms;  // SMs of the device (the persistent grids)
};

// Bytes of workspace the backward needs (two fp32 row vectors per query row,
// padded to whole 128-row tiles).
size_t bwd_workspace_bytes(int B, int Hq, int Sq);

// Kernel launchers (return cudaError_t of the launch).
cudaError_t launch_attn_bwd(const BwdLaunch& a, cudaStream_t stream);
cudaError_t launch_attn_fwd(const FwdLaunch& a, cudaStream_t stream);
// d = 256: one Q tile per CTA, two S buffers and O in tensor memory (dense,
// varlen and strided inputs; not paged).
cudaError_t launch_attn_fwd256(const FwdLaunch& a, cudaStream_t stream);
cudaError_t launch_attn_fill_empty(const FwdLaunch& a, cudaStream_t stream);
cudaError_t launch_attn_decode(const DecodeLaunch& a, cudaStream_t stream);
cudaError_t launch_wait_timeout_check(int* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace attn
