// bsa_kernels.cu - the bandwidth-bound steps around the tensor-core kernels:
//   * mask compaction (BlockSparseMask -> per-column / per-row active lists),
//     page "aclnnBlockSparseAttentionGrad", parameter table, row
//     blockSparseMaskOptional (1 = the block takes part);
//   * the backward work planner (column lists -> balanced work items);
//   * the packing of the token mask attenMask into bit rows;
//   * the preprocess D = rowsum(dOut * attentionOut) (formulas, softmax_grad)
//     and lse*log2(e), plus zeroing of the fp32 dQ accumulator;
//   * the finalize kernels: fp32 dQ (and split-column dK/dV) -> output dtype,
//     zeros for padding rows and for key tiles no query selects.
#include <algorithm>
#include <cstring>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bsa_common.h"
#include "bsa_device.cuh"
#include "bsa_launch.h"

namespace bsa {

// --------------------------------------------------------------------------
// compaction
// --------------------------------------------------------------------------
// Sub-block bits of tile (it, jt) for (b, h): bit (ri*2+cj) set when block
// (it*rb+ri, jt*cb+cj) lies inside the valid range, is selected and holds at
// least one pair that the sliding window and the token mask keep.
__device__ __forceinline__ int tile_bits(const CompactArgs& a, int b, int h, int it, int jt,
                                         int Lq, int Lk) {
  int bits = 0;
  for (int ri = 0; ri < a.rb; ++ri) {
    const int i = it * a.rb + ri;
    if ((int64_t)i * a.bx >= Lq) break;
    for (int cj = 0; cj < a.cb; ++cj) {
      const int j = jt * a.cb + cj;
      if ((int64_t)j * a.by >= Lk) break;
      bool on = true;
      if (a.has_mask) {
        on = (i < a.Mq && j < a.Mk) &&
             a.mask[(int64_t)b * a.sb + (int64_t)h * a.sh + (int64_t)i * a.si + j] != 0;
      }
      if (on && a.win)
        on = win_meets((int64_t)i * a.bx, min((int64_t)(i + 1) * a.bx, (int64_t)Lq),
                       (int64_t)j * a.by, min((int64_t)(j + 1) * a.by, (int64_t)Lk), a.win_pre,
                       a.win_next);
      if (on && a.am_sub != nullptr) on = am_block_meets(a.am_sub, a.am_sk, i, j, a.bx, a.by);
      if (on) bits |= 1 << (ri * 2 + cj);
    }
  }
  return bits;
}

// One warp per column (b, g, jt, hl) with index ((b*N2+g)*col_slots + jt)*G + hl.
// fill == 0: counts[col] = active tiles; fill == 1: writes the entries.
__device__ __forceinline__ void columns_body(const CompactArgs& a, int fill) {
  if (fill && a.zero != nullptr) {  // e.g. the fp32 slots of split columns
    const int64_t n4 = (int64_t)(*a.zero_count) * a.zero_per / 4;
    float4* z = reinterpret_cast<float4*>(a.zero);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (int64_t)gridDim.x * blockDim.x)
      z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int warps = blockDim.x >> 5;
  const int col = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int ncols = a.B * a.N2 * a.col_slots * a.G;
  if (col >= ncols) return;
  const int hl = col % a.G;
  const int r = col / a.G;
  const int jt = r % a.col_slots;
  const int bg = r / a.col_slots;
  const int g = bg % a.N2;
  const int b = bg / a.N2;
  const int h = g * a.G + hl;
  const int Lq = a.lq[b], Lk = a.lk[b];
  const int nrows = (Lq + a.tq - 1) / a.tq;
  const int ncolt = (Lk + a.tk - 1) / a.tk;
  int count = 0;
  int base = fill ? a.ptr[col] : 0;
  if (jt < ncolt) {
    for (int it0 = 0; it0 < nrows; it0 += 32) {
      const int it = it0 + lane;
      const int bits = it < nrows ? tile_bits(a, b, h, it, jt, Lq, Lk) : 0;
      const unsigned ball = __ballot_sync(0xffffffffu, bits != 0);
      if (fill && bits) {
        const int pos = base + count + __popc(ball & ((1u << lane) - 1u));
        if (kChecks && a.out_cap > 0 && pos >= a.out_cap) check_failed(a.check_hdr, kCheckEntryPos);
        else a.out[pos] = a.plain ? it : pack_entry(it, hl, bits);
      }
      count += __popc(ball);
    }
  }
  if (!fill && lane == 0) a.counts[col] = count;
  // the test of the checks: column 0's first entry names a query tile past the last one
  if (kChecks && fill && a.check_test && col == 0 && lane == 0 && count > 0)
    a.out[base] = pack_entry(a.row_slots, 0, 1);
}

__global__ void k_columns(CompactArgs a, int fill) {
  columns_body(a, fill);
}

// The column count of a backward run with the per-batch arrays inline: block 0
// also stores them into the workspace for the kernels after this one.
__global__ void k_columns_info(CompactArgs a, const __grid_constant__ InfoInline info) {
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < info.n; i += blockDim.x) info.dst[i] = info.v[i];
  a.lq = info.v + info.off[0];
  a.lk = info.v + info.off[1];
  columns_body(a, 0);
}

// One warp per row (b, h, it) with index (b*N1+h)*row_slots + it.
__global__ void k_rows(CompactArgs a, int fill) {
  const int warps = blockDim.x >> 5;
  const int row = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int nrows_all = a.B * a.N1 * a.row_slots;
  if (row >= nrows_all) return;
  const int it = row % a.row_slots;
  const int bh = row / a.row_slots;
  const int h = bh % a.N1;
  const int b = bh / a.N1;
  const int Lq = a.lq[b], Lk = a.lk[b];
  const int nrows = (Lq + a.tq - 1) / a.tq;
  const int ncolt = (Lk + a.tk - 1) / a.tk;
  int count = 0;
  int base = fill ? a.ptr[row] : 0;
  if (it < nrows) {
    for (int jt0 = 0; jt0 < ncolt; jt0 += 32) {
      const int jt = jt0 + lane;
      const int bits = jt < ncolt ? tile_bits(a, b, h, it, jt, Lq, Lk) : 0;
      const unsigned ball = __ballot_sync(0xffffffffu, bits != 0);
      if (fill && bits) {
        const int pos = base + count + __popc(ball & ((1u << lane) - 1u));
        a.out[pos] = a.plain ? jt : pack_entry(jt, 0, bits);
      }
      count += __popc(ball);
    }
  }
  if (!fill && lane == 0) a.counts[row] = count;
}

// --------------------------------------------------------------------------
// token mask packing (attenMaskOptional; 1 = the pair is masked out)
// --------------------------------------------------------------------------
// One 256-thread block per strip of kAmStrip 64x64 sub-blocks (i, j0 ..
// j0 + kAmStrip - 1), out as two 32-bit words per query row and sub-block
// (keys 64j .. 64j+63), two per key row (queries 64i .. 64i+63) and each
// sub-block's class. Positions outside the matrix count as masked. Thread
// (r, q) reads 16 bytes of row r (16-byte loads from a row-contiguous, 16-byte
// aligned matrix, all of its loads in flight at once; else byte by byte
// through shared memory) and packs them to 16 bits in registers; the key-row
// words come from 32x32 bit transposes by warp shuffles.
constexpr int kAmStrip = 4;

// Four 0/1 bytes of a word -> four bits (byte k -> bit k): the multiplier puts
// byte k's bit at bit 21 + k and no two partial products share a bit.
__device__ __forceinline__ uint32_t flag_nibble(uint32_t w) { return ((w * 0x00204081u) >> 21) & 0xFu; }

__global__ void __launch_bounds__(256) k_amask(AmaskArgs a) {
  __shared__ __align__(16) uint8_t tile[64][80];  // the byte-by-byte path, one sub-block at a time
  __shared__ uint32_t rw[kAmStrip][64][2];        // [sub-block][row][32-key half] row words
  const int i = blockIdx.y, j0 = blockIdx.x * kAmStrip, tid = threadIdx.x;
  const int r = tid >> 2, q = tid & 3, lane = tid & 31, warp = tid >> 5;
  const bool aligned = a.st1 == 1 && (a.st0 & 15) == 0 &&
                       (reinterpret_cast<uintptr_t>(a.m) & 15) == 0 && (i + 1) * 64 <= a.rows;
  uint4 u[kAmStrip];
#pragma unroll
  for (int jj = 0; jj < kAmStrip; ++jj) {
    const int j = j0 + jj;
    if (aligned && j < a.nsub_k && (j + 1) * 64 <= a.cols)
      u[jj] = *reinterpret_cast<const uint4*>(a.m + (int64_t)(i * 64 + r) * a.st0 + j * 64 + 16 * q);
  }
  uint32_t rb[kAmStrip];  // bits 16q .. 16q+15 of row r of each sub-block
#pragma unroll
  for (int jj = 0; jj < kAmStrip; ++jj) {
    const int j = j0 + jj;
    rb[jj] = 0xFFFFu;
    if (j >= a.nsub_k) continue;  // the same for the whole block
    if (aligned && (j + 1) * 64 <= a.cols) {
      uint32_t w[4] = {u[jj].x, u[jj].y, u[jj].z, u[jj].w};
      uint32_t bits = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // each byte -> 0 or 1 (bit 0 ORs the byte's bits)
        uint32_t x = w[k];
        x |= x >> 4;
        x |= x >> 2;
        x |= x >> 1;
        bits |= flag_nibble(x & 0x01010101u) << (4 * k);
      }
      rb[jj] = bits;
    } else {
      __syncthreads();  // the previous sub-block's reads of `tile` are done
      for (int e = tid; e < 64 * 64; e += 256) {
        const int rr = e >> 6, c = e & 63;
        const int s = i * 64 + rr, t = j * 64 + c;
        uint8_t v = 1;
        if (s < a.rows && t < a.cols) v = a.m[(int64_t)s * a.st0 + (int64_t)t * a.st1] != 0;
        tile[rr][c] = v;
      }
      __syncthreads();
      uint32_t bits = 0;
#pragma unroll
      for (int k = 0; k < 16; ++k) bits |= (uint32_t)tile[r][16 * q + k] << k;
      rb[jj] = bits;
    }
    const uint32_t hi = __shfl_down_sync(0xffffffffu, rb[jj], 1);
    if ((q & 1) == 0) {
      const uint32_t word = rb[jj] | (hi << 16);  // keys 32 (q/2) .. 32 (q/2) + 31 of row r
      rw[jj][r][q >> 1] = word;
      if (a.row_bits != nullptr) a.row_bits[(int64_t)(i * 64 + r) * a.wk + 2 * j + (q >> 1)] = word;
    }
  }
  __syncthreads();
  if (a.col_bits != nullptr) {
    // warp w: the 32x32 block of rows 32 rh .. and keys 32 ch .. of sub-blocks
    // w/4, w/4 + 2; lane L starts with row 32 rh + L and ends with key 32 ch + L
    const int rh = warp & 1, ch = (warp >> 1) & 1;
    for (int jj = warp >> 2; jj < kAmStrip; jj += 2) {
      const int j = j0 + jj;
      if (j >= a.nsub_k) break;
      uint32_t x = rw[jj][32 * rh + lane][ch];
#pragma unroll
      for (int sh = 16; sh >= 1; sh >>= 1) {
        const uint32_t m = sh == 16 ? 0x0000FFFFu
                         : sh == 8  ? 0x00FF00FFu
                         : sh == 4  ? 0x0F0F0F0Fu
                         : sh == 2  ? 0x33333333u
                                    : 0x55555555u;  // keys whose bit `sh` is clear
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, sh);
        x = (lane & sh) ? ((x & ~m) | ((y & ~m) >> sh)) : ((x & m) | ((y & m) << sh));
      }
      a.col_bits[(int64_t)(j * 64 + 32 * ch + lane) * a.wq + 2 * i + rh] = x;
    }
  }
#pragma unroll
  for (int jj = 0; jj < kAmStrip; ++jj) {
    const int j = j0 + jj;
    if (j >= a.nsub_k) break;
    const int all = __syncthreads_and(rb[jj] == 0xFFFFu);
    const int any = __syncthreads_or(rb[jj] != 0u);
    if (tid == 0) a.sub[(int64_t)i * a.nsub_k + j] = all ? kAmAll : (any ? kAmSome : kAmNone);
  }
}

// Block-wide exclusive scan of one value per thread (1024 threads).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[w] = x;
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    int s = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nw) warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int warp_prefix = w ? warp_sums[w - 1] : 0;
  const int res = warp_prefix + x - v;
  const int tot = warp_sums[(blockDim.x >> 5) - 1];
  __syncthreads();
  *total = tot;
  return res;
}

// out[i] = sum_{k<i} in[k] for i in [0, n]; single block of 1024 threads.
__global__ void k_scan(const int* in, int* out, int n) {
  __shared__ int ws[32];
  int carry = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const int v = i < n ? in[i] : 0;
    int tot;
    const int ex = block_exclusive_scan(v, ws, &tot);
    if (i < n) out[i] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) out[n] = carry;
}

// Backward planner (single block of 1024 threads):
//  1. colptr = exclusive scan of the grouped column counts;
//  2. per key tile gc (all G heads of the group): n = its active tiles; a
//     column longer than the chunk length of its wave (and while partial
//     slots remain) is split into balanced chunks that add into an fp32 slot;
//  3. items are ordered by wave, longest first within a wave (counting sort
//     on the item length), so the persistent CTAs pick the long work of a
//     wave before its short work.
__device__ __forceinline__ int chunk_begin(int n, int chunks, int c) {
  return (int)(((int64_t)c * n) / chunks);
}

__global__ void __launch_bounds__(1024) k_plan(Plan p) {
  if (threadIdx.x == 0) {  // the error words of the run (before any check of this kernel)
    p.header[kHdrError] = 0;
    p.header[kHdrErrorWhere] = 0;
    p.header[kHdrCheckWhere] = 0;
    for (int i = 0; i < 16; ++i) p.header[kHdrErrorCounts + i] = 0;
  }
  // Items are ordered by (wave, length descending): a wave is a run of
  // consecutive (b, kv head) groups (p.n_waves of them, equal counts), and
  // within a wave the longest items go first. Lengths >= kLenB - 1 share a
  // bucket.
  constexpr int kLenB = 64, kMaxWaves = 32, kKeys = kLenB * kMaxWaves;
  __shared__ int ws[32];
  __shared__ int s_L;
  __shared__ int hist[kKeys];
  const int nbg = p.NGC / p.Mk_t;
  auto wave_of = [&](int gc) { return (int)((int64_t)(gc / p.Mk_t) * p.n_waves / nbg); };
  auto key_of = [&](int gc, int len) {
    return wave_of(gc) * kLenB + (kLenB - 1 - min(len, kLenB - 1));
  };
  int carry = 0;
  for (int base = 0; base < p.NC; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const int v = i < p.NC ? p.colcnt[i] : 0;
    int tot;
    const int ex = block_exclusive_scan(v, ws, &tot);
    if (i < p.NC) p.colptr[i] = carry + ex;
    carry += tot;
  }
  const int T = carry;
  if (threadIdx.x == 0) {
    p.colptr[p.NC] = T;
    int L = (T + 2 * p.num_sms - 1) / (2 * p.num_sms);
    if (L < p.min_chunk) L = p.min_chunk;
    s_L = L;
  }
  for (int i = threadIdx.x; i < kKeys; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int L = s_L;
  // Chunk length of key tile gc: an item claimed when its wave starts must end
  // before the work left from there on is done, so the chunks shrink wave by
  // wave, to half an SM's share of one wave in the last (a long item claimed
  // late would otherwise run on alone while the other SMs idle).
  auto chunk_len = [&](int gc) {
    const int64_t den = (int64_t)p.n_waves * 2 * p.num_sms;
    const int64_t left = (int64_t)(p.n_waves - wave_of(gc)) * T;
    return max((int)((left + den - 1) / den), p.min_chunk);
  };
  // pass 1: split decision, slots, length histogram (descending buckets), and
  // the list of key tiles the finalize kernel writes (no entries, or split).
  // Key tiles are taken from the last one back, so that when slots run short
  // the late waves, whose long items would end the kernel, still split.
  int slot_carry = 0, fin_carry = 0;
  for (int base = 0; base < p.NGC; base += blockDim.x) {
    const int r = base + threadIdx.x;
    const bool valid = r < p.NGC;
    const int gc = p.NGC - 1 - r;
    int n = 0, Lw = L;
    if (valid) {
      n = p.colptr[(gc + 1) * p.G] - p.colptr[gc * p.G];
      Lw = chunk_len(gc);
    }
    const int want = (valid && n > Lw) ? 1 : 0;
    int tot;
    const int sidx = block_exclusive_scan(want, ws, &tot) + slot_carry;
    slot_carry += tot;
    const int split = want && (sidx < p.max_slots);
    const int fin = valid && (n == 0 || split);
    const int fidx = block_exclusive_scan(fin, ws, &tot) + fin_carry;
    fin_carry += tot;
    if (fin) p.fin_tiles[fidx] = gc;
    if (valid) {
      p.colinfo[gc] = (n == 0) ? -1 : (split ? sidx : -2);
      const int chunks = split ? (n + Lw - 1) / Lw : (n > 0 ? 1 : 0);
      for (int c = 0; c < chunks; ++c) {
        const int len = chunk_begin(n, chunks, c + 1) - chunk_begin(n, chunks, c);
        atomicAdd(&hist[key_of(gc, len)], 1);
      }
    }
  }
  __syncthreads();
  int total_items = 0;
  for (int base = 0; base < kKeys; base += blockDim.x) {  // bucket start offsets
    const int v = hist[base + threadIdx.x];
    int tot;
    const int ex = block_exclusive_scan(v, ws, &tot);
    hist[base + threadIdx.x] = total_items + ex;
    total_items += tot;
  }
  __syncthreads();
  // pass 2: place the items
  for (int base = 0; base < p.NGC; base += blockDim.x) {
    const int gc = base + threadIdx.x;
    if (gc >= p.NGC) continue;
    const int info = p.colinfo[gc];
    if (info == -1) continue;
    const int e0 = p.colptr[gc * p.G];
    const int n = p.colptr[(gc + 1) * p.G] - e0;
    const int Lw = chunk_len(gc);
    const int chunks = info >= 0 ? (n + Lw - 1) / Lw : 1;
    for (int c = 0; c < chunks; ++c) {
      const int b0 = chunk_begin(n, chunks, c), b1 = chunk_begin(n, chunks, c + 1);
      const int pos = atomicAdd(&hist[key_of(gc, b1 - b0)], 1);
      if (kChecks && pos >= p.max_items) check_failed(p.header, kCheckItemPos);
      else p.items[pos] = make_int4(gc, e0 + b0, e0 + b1, info >= 0 ? info : -1);
    }
  }
  if (threadIdx.x == 0) {
    p.header[kHdrNumItems] = total_items;
    p.header[kHdrTotalTiles] = T;
    p.header[kHdrSlotsUsed] = min(slot_carry, p.max_slots);
    p.header[kHdrFinTiles] = fin_carry;
    p.header[kHdrChunkLen] = L;
    p.header[kHdrWorkCounter] = 0;
    p.header[kHdrDqCounter] = 0;
  }
}

// --------------------------------------------------------------------------
// preprocess: D_s = sum_d dout_sd * out_sd, lse2_s = lse_s * log2(e); zero dQacc
// --------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float2 to_f2(uint32_t u);
template <>
__device__ __forceinline__ float2 to_f2<__nv_bfloat16>(uint32_t u) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(h);
}
template <>
__device__ __forceinline__ float2 to_f2<__half>(uint32_t u) {
  __half2 h = *reinterpret_cast<__half2*>(&u);
  return __half22float2(h);
}

template <typename T, int D>
__global__ void __launch_bounds__(256) k_preprocess(Plan p, const __grid_constant__ InfoInline info) {
  if (info.n > 0) {  // the per-batch arrays from the parameter, not the workspace
    p.lq = info.v + info.off[0];
    p.cu_q = info.v + info.off[2];
    p.qrow = info.v + info.off[4];
    p.qtile_b = info.v + info.off[6];
  }
  constexpr int TPR = D / 8;  // threads per row, 8 elements (16 B) each
  constexpr int RPB = 256 / TPR;
  const int sub = threadIdx.x % TPR;
  const int64_t row = (int64_t)blockIdx.x * RPB + threadIdx.x / TPR;  // over N1 * Rq
  if (row >= (int64_t)p.N1 * p.Rq) return;
  const int h = (int)(row / p.Rq);
  const int r = (int)(row % p.Rq);
  const int b = p.qtile_b[r / kTile];
  const int s = r - p.qrow[b];
  const bool valid = s < p.lq[b];
  float acc = 0.f;
  if (valid) {
    int64_t off;
    if (p.layout == kLayoutBNSD)
      off = (((int64_t)b * p.N1 + h) * p.Sq + s) * D;
    else
      off = (((int64_t)p.cu_q[b] + s) * p.N1 + h) * D;
    const uint4 a = reinterpret_cast<const uint4*>(static_cast<const T*>(p.dout) + off)[sub];
    const uint4 c = reinterpret_cast<const uint4*>(static_cast<const T*>(p.out) + off)[sub];
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 x = to_f2<T>(av[k]), y = to_f2<T>(cv[k]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  }
#pragma unroll
  for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, TPR);
  if (sub == 0) {
    // rows past the query length: +inf, so that P = exp2(x - lse2) is exactly
    // zero in their columns of the backward
    float l2 = __int_as_float(0x7f800000);
    if (valid) {
      int64_t li;
      if (p.layout == kLayoutBNSD)
        li = ((int64_t)b * p.N1 + h) * p.Sq + s;
      else
        li = ((int64_t)p.cu_q[b] + s) * p.N1 + h;
      l2 = p.lse[li] * 1.4426950408889634f;
    }
    p.dvec[row] = valid ? acc : 0.f;
    p.lse2[row] = l2;
  }
  if (!p.det) {  // the deterministic dQ pass does not use the accumulator
    float4* dst = reinterpret_cast<float4*>(p.dqacc + row * D) + sub * 2;
    dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// --------------------------------------------------------------------------
// finalize
// --------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <typename T>
__device__ __forceinline__ T cvt1(float a);
template <>
__device__ __forceinline__ __nv_bfloat16 cvt1<__nv_bfloat16>(float a) {
  return __float2bfloat16_rn(a);
}
template <>
__device__ __forceinline__ __half cvt1<__half>(float a) {
  return __float2half_rn(a);
}

// Writes 8 consecutive (in d) output values at element offset `off` with
// element stride `sd`: one 16-byte store when `vec`, else scalar stores.
template <typename T>
__device__ __forceinline__ void store8(void* base, int64_t off, int64_t sd, bool vec,
                                       const float (&x)[8]) {
  T* p = static_cast<T*>(base) + off;
  if (vec) {
    uint4 u;
    u.x = pack2<T>(x[0], x[1]);
    u.y = pack2<T>(x[2], x[3]);
    u.z = pack2<T>(x[4], x[5]);
    u.w = pack2<T>(x[6], x[7]);
    *reinterpret_cast<uint4*>(p) = u;
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) p[k * sd] = cvt1<T>(x[k]);
  }
}

__device__ __forceinline__ int batch_of_token(const int* cu, int B, int tok) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= tok) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// dq[b,h,s,:] = scale * dQacc (0 on padding rows), any output strides.
template <typename T, int D>
__device__ __forceinline__ void finalize_dq_rows(const Plan& p) {
  constexpr int TPR = D / 8;
  constexpr int RPB = 256 / TPR;
  constexpr int kRows = 4;  // rows per thread and pass: their loads are in flight together
  const int sub = threadIdx.x % TPR;
  const int64_t nrows = (p.layout == kLayoutBNSD) ? (int64_t)p.B * p.N1 * p.Sq
                                                  : (int64_t)p.Tq * p.N1;
  const int64_t stride = (int64_t)gridDim.x * RPB;
  const int64_t sd = p.dq_st[p.layout == kLayoutBNSD ? 3 : 2];
  for (int64_t row0 = (int64_t)blockIdx.x * RPB + threadIdx.x / TPR; row0 < nrows;
       row0 += kRows * stride) {
    int64_t off[kRows];
    const float* acc[kRows];  // null: a padding row (zeros)
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      const int64_t row = row0 + u * stride;
      acc[u] = nullptr;
      off[u] = -1;
      if (row >= nrows) continue;
      int b, h, s;
      if (p.layout == kLayoutBNSD) {
        s = (int)(row % p.Sq);
        const int64_t bh = row / p.Sq;
        h = (int)(bh % p.N1);
        b = (int)(bh / p.N1);
        off[u] = b * p.dq_st[0] + h * p.dq_st[1] + s * p.dq_st[2];
      } else {
        h = (int)(row % p.N1);
        const int tok = (int)(row / p.N1);
        b = batch_of_token(p.cu_q, p.B, tok);
        s = tok - p.cu_q[b];
        off[u] = tok * p.dq_st[0] + h * p.dq_st[1];
      }
      if (s < p.lq[b]) acc[u] = p.dqacc + ((int64_t)h * p.Rq + p.qrow[b] + s) * D + sub * 8;
    }
    float4 a[kRows], c[kRows];
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      a[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      c[u] = a[u];
      if (acc[u] != nullptr) {
        a[u] = reinterpret_cast<const float4*>(acc[u])[0];
        c[u] = reinterpret_cast<const float4*>(acc[u])[1];
      }
    }
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      if (off[u] < 0) continue;
      const float x[8] = {a[u].x * p.scale, a[u].y * p.scale, a[u].z * p.scale, a[u].w * p.scale,
                          c[u].x * p.scale, c[u].y * p.scale, c[u].z * p.scale, c[u].w * p.scale};
      store8<T>(p.dq, off[u] + sub * 8 * sd, sd, p.dq_vec != 0, x);
    }
  }
}

// dk/dv rows of the key tiles the backward kernel did not write (the list
// fin_tiles from the planner): zeros for tiles no query selects, the fp32 slot
// (dK already scaled) for split tiles.
template <typename T, int D>
__device__ __forceinline__ void finalize_dkdv_tiles(const Plan& p) {
  constexpr int TPR = D / 8;
  constexpr int RPB = 256 / TPR;
  const int sub = threadIdx.x % TPR;
  const int64_t nrows = (int64_t)p.header[kHdrFinTiles] * kTile;
  for (int64_t row = (int64_t)blockIdx.x * RPB + threadIdx.x / TPR; row < nrows;
       row += (int64_t)gridDim.x * RPB) {
    const int gc = p.fin_tiles[row / kTile];
    if (kChecks && !(gc >= 0 && gc < p.NGC && p.colinfo[gc] < p.max_slots)) {
      check_failed(p.header, kCheckFinTile);
      continue;
    }
    const int jt = gc % p.Mk_t;
    const int bg = gc / p.Mk_t;
    const int g = bg % p.N2, b = bg / p.N2;
    const int t = jt * kTile + (int)(row % kTile);
    int64_t ok, ov;
    if (p.layout == kLayoutBNSD) {
      if (t >= p.Skv) continue;
      ok = b * p.dk_st[0] + g * p.dk_st[1] + t * p.dk_st[2];
      ov = b * p.dv_st[0] + g * p.dv_st[1] + t * p.dv_st[2];
    } else {
      if (t >= p.lk[b]) continue;
      const int64_t tok = (int64_t)p.cu_k[b] + t;
      ok = tok * p.dk_st[0] + g * p.dk_st[1];
      ov = tok * p.dv_st[0] + g * p.dv_st[1];
    }
    const int info = p.colinfo[gc];
    float xk[8], xv[8];
    if (info >= 0 && t < p.lk[b]) {
      const float* sl = p.slots + (int64_t)info * 2 * kTile * D;
      const float4* sk = reinterpret_cast<const float4*>(sl + (t % kTile) * D + sub * 8);
      const float4* sv = reinterpret_cast<const float4*>(sl + (kTile + t % kTile) * D + sub * 8);
      const float4 a = sk[0], c = sk[1], e = sv[0], f = sv[1];
      xk[0] = a.x; xk[1] = a.y; xk[2] = a.z; xk[3] = a.w;
      xk[4] = c.x; xk[5] = c.y; xk[6] = c.z; xk[7] = c.w;
      xv[0] = e.x; xv[1] = e.y; xv[2] = e.z; xv[3] = e.w;
      xv[4] = f.x; xv[5] = f.y; xv[6] = f.z; xv[7] = f.w;
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) xk[k] = xv[k] = 0.f;
    }
    const int li = p.layout == kLayoutBNSD ? 3 : 2;
    store8<T>(p.dk, ok + sub * 8 * p.dk_st[li], p.dk_st[li], p.dkv_vec != 0, xk);
    store8<T>(p.dv, ov + sub * 8 * p.dv_st[li], p.dv_st[li], p.dkv_vec != 0, xv);
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(256) k_finalize(Plan p) {
  if (!p.det) finalize_dq_rows<T, D>(p);  // else dQ came from the deterministic pass
  finalize_dkdv_tiles<T, D>(p);
}

// --------------------------------------------------------------------------
// small host arrays into device memory through kernel parameters (no copy
// from pageable memory, which would first synchronize the stream)
// --------------------------------------------------------------------------
template <int N>
struct UploadBuf {
  int v[N];
};
template <int N>
__global__ void k_upload(UploadBuf<N> u, int n, int* dst) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = u.v[i];
}
template <int N>
static cudaError_t upload_t(const int* host, int n, int* dst, cudaStream_t st) {
  UploadBuf<N> u;
  std::memcpy(u.v, host, sizeof(int) * n);
  k_upload<N><<<1, 256, 0, st>>>(u, n, dst);
  return cudaGetLastError();
}
cudaError_t launch_upload(const int* host, int n, int* dst, cudaStream_t st) {
  // longer arrays go in several launches of 7680 ints (30 KB of parameters)
  // each, so the caller's host array is never read after the call returns
  // (stream capture records the parameters by value)
  while (n > 7680) {
    const cudaError_t e = upload_t<7680>(host, 7680, dst, st);
    if (e != cudaSuccess) return e;
    host += 7680;
    dst += 7680;
    n -= 7680;
  }
  if (n <= 0) return cudaSuccess;
  if (n <= 256) return upload_t<256>(host, n, dst, st);
  if (n <= 2048) return upload_t<2048>(host, n, dst, st);
  return upload_t<7680>(host, n, dst, st);
}

// --------------------------------------------------------------------------
// launchers
// --------------------------------------------------------------------------
cudaError_t launch_columns(const CompactArgs& a, int fill, cudaStream_t st,
                           const InfoInline* info) {
  const int ncols = a.B * a.N2 * a.col_slots * a.G;
  if (info != nullptr && info->n > 0 && !fill) {
    // block 0 stores the per-batch arrays, so the launch has one even with no column
    k_columns_info<<<std::max((ncols + 7) / 8, 1), 256, 0, st>>>(a, *info);
    return cudaGetLastError();
  }
  if (ncols == 0) return cudaSuccess;
  k_columns<<<(ncols + 7) / 8, 256, 0, st>>>(a, fill);
  return cudaGetLastError();
}

cudaError_t launch_amask(const AmaskArgs& a, cudaStream_t st) {
  if (a.nsub_q == 0 || a.nsub_k == 0) return cudaSuccess;
  k_amask<<<dim3((a.nsub_k + kAmStrip - 1) / kAmStrip, a.nsub_q), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rows(const CompactArgs& a, int fill, cudaStream_t st) {
  const int nrows = a.B * a.N1 * a.row_slots;
  if (nrows == 0) return cudaSuccess;
  k_rows<<<(nrows + 7) / 8, 256, 0, st>>>(a, fill);
  return cudaGetLastError();
}

cudaError_t launch_scan(const int* in, int* out, int n, cudaStream_t st) {
  k_scan<<<1, 1024, 0, st>>>(in, out, n);
  return cudaGetLastError();
}

cudaError_t launch_plan(const Plan& p, cudaStream_t st) {
  k_plan<<<1, 1024, 0, st>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t launch_pre_t(const Plan& p, cudaStream_t st, const InfoInline& info) {
  constexpr int RPB = 256 / (D / 8);
  const int64_t rows = (int64_t)p.N1 * p.Rq;
  if (rows == 0) return cudaSuccess;
  k_preprocess<T, D><<<(unsigned)((rows + RPB - 1) / RPB), 256, 0, st>>>(p, info);
  return cudaGetLastError();
}

cudaError_t launch_preprocess(const Plan& p, cudaStream_t st, const InfoInline* info) {
  static const InfoInline none = {};  // n = 0: the workspace copy
  const InfoInline& in = info != nullptr ? *info : none;
  if (p.dtype == kDtBF16)
    return p.D == 128 ? launch_pre_t<__nv_bfloat16, 128>(p, st, in)
                      : launch_pre_t<__nv_bfloat16, 64>(p, st, in);
  return p.D == 128 ? launch_pre_t<__half, 128>(p, st, in) : launch_pre_t<__half, 64>(p, st, in);
}

template <typename T, int D>
static cudaError_t launch_fin_t(const Plan& p, cudaStream_t st) {
  const int grid = p.num_sms * 8;
  k_finalize<T, D><<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const Plan& p, cudaStream_t st) {
  if (p.dtype == kDtBF16)
    return p.D == 128 ? launch_fin_t<__nv_bfloat16, 128>(p, st)
                      : launch_fin_t<__nv_bfloat16, 64>(p, st);
  return p.D == 128 ? launch_fin_t<__half, 128>(p, st) : launch_fin_t<__half, 64>(p, st);
}

}  // namespace bsa
