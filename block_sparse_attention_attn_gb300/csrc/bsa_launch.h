// bsa_launch.h - host-side launchers of the kernels (all asynchronous on `st`).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "bsa_common.h"

namespace bsa {

// Arguments of the mask compaction kernels. Columns are indexed
// ((b*N2 + g)*col_slots + jt)*G + hl, rows (b*N1 + h)*row_slots + it; slots
// past the valid tiles of a batch get count 0 (so a slot count of Mq+1 / Mk+1
// yields the CSR/CSC pointer layout with a closing entry per (b, h)).
struct CompactArgs {
  const uint8_t* mask;
  int64_t sb, sh, si;  // mask strides (j stride 1)
  int has_mask;
  int B, N1, N2, G;
  int Mq, Mk;          // mask dims in blocks
  int bx, by, rb, cb;  // block shape and blocks per tile
  int tq, tk;          // tile size in tokens (rb*bx, cb*by)
  int col_slots, row_slots;
  const int* lq;       // device, per batch
  const int* lk;
  int* counts;         // count pass output
  const int* ptr;      // fill pass: exclusive scan of counts
  int32_t* out;        // fill pass output
  int plain;           // 1: store the tile index only; 0: packed entry
  int win;             // drop sub-blocks outside the sliding window (Plan::win)
  int64_t win_pre, win_next;
  const uint8_t* am_sub;  // drop blocks the token mask masks entirely (or null)
  int am_sk;
  float* zero;            // fill pass: optional fp32 region cleared first (or null)
  const int* zero_count;  // device: number of zero_per-float units to clear
  int zero_per;           // floats per unit, a multiple of 4
  // bounds-check variant only: entries past out_cap (0: unchecked) are dropped
  // and recorded in check_hdr; check_test plants one out-of-range entry in
  // column 0 (the test of the checks)
  int* check_hdr;
  int out_cap;
  int check_test;
};

// Sets the thread's bsa_last_error() text (used by entry points outside bsa_api.cpp).
void set_last_error(const char* msg);

// n ints from host memory to dst, through kernel parameters (one launch per
// 7680 ints): the host array may be reused as soon as the call returns, and
// the upload can be captured in a CUDA graph.
cudaError_t launch_upload(const int* host, int n, int* dst, cudaStream_t st);

// The per-batch arrays of a run (Plan::lq .. Plan::qtile_b) inline in a kernel
// parameter, for the two kernels that start a backward run side by side (the
// column count and the preprocess): neither waits for an upload launch, and
// the column count copies them to `dst` in the workspace for the kernels that
// come after it.
constexpr int kInfoInline = 1024;
struct InfoInline {
  int n;        // ints in v; 0: none (the kernels read the workspace copy)
  int off[7];   // offsets of lq, lk, cu_q, cu_k, qrow, krow, qtile_b in v
  int* dst;     // the workspace copy
  int v[kInfoInline];
};

// Column count (fill = 0) or fill (fill = 1) over the mask. `info` (count
// only): the per-batch arrays inline, copied to info->dst.
cudaError_t launch_columns(const CompactArgs& a, int fill, cudaStream_t st,
                           const InfoInline* info = nullptr);

// Packing of the token mask attenMask [rows, cols] (element strides st0, st1;
// nonzero = masked) into the bit rows and sub-block classes of Plan::am_*.
struct AmaskArgs {
  const uint8_t* m;
  int64_t st0, st1;
  int rows, cols;
  uint32_t* row_bits;  // [nsub_q*64][wk] (null: not written)
  uint32_t* col_bits;  // [nsub_k*64][wq] (null: not written)
  uint8_t* sub;        // [nsub_q][nsub_k]
  int nsub_q, nsub_k;  // 64x64 sub-blocks (2 * tiles each way)
  int wk, wq;          // words per bit row (2*nsub_k, 2*nsub_q)
};
cudaError_t launch_amask(const AmaskArgs& a, cudaStream_t st);
cudaError_t launch_rows(const CompactArgs& a, int fill, cudaStream_t st);
cudaError_t launch_scan(const int* in, int* out, int n, cudaStream_t st);
cudaError_t launch_plan(const Plan& p, cudaStream_t st);
cudaError_t launch_preprocess(const Plan& p, cudaStream_t st, const InfoInline* info = nullptr);
cudaError_t launch_finalize(const Plan& p, cudaStream_t st);

// Tensor maps of the backward / forward kernels (3-D views, 64-element x 128-row
// boxes, 128-byte swizzle): BNSD (d, s, b*N+h), TND (d, h, token).
struct BwdMaps {
  CUtensorMap q, k, v, dout;
  CUtensorMap dqacc;  // fp32 [N1*Rq rows, D], box 32 x 32, 128-byte swizzle (reduce-add)
  CUtensorMap dk, dv; // outputs, box 64 x 32 rows, 128-byte swizzle: BNSD (d, s, n, b), TND (d, n, t)
  CUtensorMap k64, v64; // K, V with 64-row boxes (the 64-key-block kernel only)
};
cudaError_t launch_bwd(const Plan& p, const BwdMaps& m, cudaStream_t st);
// Backward for key blocks of 64 tokens with D = 128 and no element masks
// (query-major tiles, one pass per key block of a 128-key tile).
bool bwd_k64_applies(const Plan& p);
cudaError_t launch_bwd_k64(const Plan& p, const BwdMaps& m, cudaStream_t st);
// Deterministic dQ pass (query-tile stationary), used when p.det is set.
cudaError_t launch_bwd_dq(const Plan& p, const BwdMaps& m, cudaStream_t st);
size_t bwd_smem_bytes(int D);

struct FwdMaps {
  CUtensorMap q, k, v;
};
struct FwdPlan {
  Plan p;          // shared geometry and tensors (out -> p.dq slot unused)
  void* out;       // attentionOut
  float* lse_out;  // softmaxLse
  int64_t out_st[4];
  int64_t lse_st[3];
  int out_vec;
  int n_rows_items; // B * N1 * (BNSD: ceil(Sq/128), TND: Mq_t)
};
cudaError_t launch_fwd(const FwdPlan& f, const FwdMaps& m, cudaStream_t st);
size_t fwd_smem_bytes(int D);

}  // namespace bsa
