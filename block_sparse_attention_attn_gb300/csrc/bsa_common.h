// bsa_common.h - plan structures shared by the host planner and the kernels.
//
// Terminology (aclnnBlockSparseAttentionGrad page, parameter table):
//   B batch, N1 query heads, N2 = numKeyValueHeads, G = N1/N2, D head dim,
//   bx/by = blockShape (query / key direction), Mq/Mk = mask block counts.
// The kernels work on 128x128 token tiles: a tile holds rb = 128/bx query
// blocks and cb = 128/by key blocks (1 or 2 each); a tile takes part when any
// of its blocks is selected, and the blocks it holds but that are not selected
// are masked out element by element ("sub-block mask", 4 bits).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace bsa {

constexpr int kTile = 128;            // tile rows (query and key direction)
constexpr int kLayoutBNSD = 0;
constexpr int kLayoutTND = 1;
constexpr int kDtF16 = 1;
constexpr int kDtBF16 = 2;

// header words at the start of every workspace
enum HeaderWord {
  kHdrError = 0,       // nonzero: a kernel gave up (bounded wait / bad state)
  kHdrWorkCounter = 1, // persistent-kernel work queue head
  kHdrNumItems = 2,    // number of backward work items
  kHdrTotalTiles = 3,  // active tiles
  kHdrSlotsUsed = 4,   // split columns that got an fp32 partial slot
  kHdrChunkLen = 5,    // split threshold used
  kHdrErrorWhere = 6,  // code of the first wait that gave up
  kHdrFinTiles = 7,    // key tiles the finalize kernel writes (unselected or split)
  kHdrDqCounter = 8,   // work-queue head of the deterministic dQ pass
  kHdrCheckWhere = 9,  // bounds-check build: id of the first check that failed
  kHdrErrorCounts = 16, // [16, 32): number of failed waits per code
  kHdrWords = 64
};

// Error codes written to kHdrErrorWhere (first failure wins).
enum ErrWhere {
  kErrNone = 0,
  kErrSmemAlign = 1,
  kErrWaitItem = 2,
  kErrWaitKV = 3,
  kErrWaitQ = 4,
  kErrWaitS = 5,
  kErrWaitDP = 6,
  kErrWaitP = 7,
  kErrWaitDS = 8,
  kErrWaitDQ = 9,
  kErrWaitAcc = 10,
  kErrWaitMisc = 11,
  kErrWaitTest = 12,     // the deliberate wait of the wait_test switch
  kErrBounds = 13,       // bounds-check build: an index outside its array (see kHdrCheckWhere)
};

// Checks of the bounds-check build (kHdrCheckWhere).
enum CheckId {
  kCheckItem = 1,        // a work item: key tile, entry range or slot out of range
  kCheckEntry = 2,       // a list entry: query tile or local head out of range
  kCheckItemPos = 3,     // the planner placing an item past the item list
  kCheckEntryPos = 4,    // the fill placing an entry past the entry list
  kCheckFinTile = 5,     // the finalize list naming a key tile or slot out of range
};

// Entry of a backward work list: query tile `it` of local head `hl`, with the
// sub-block mask in bits 28..31 (bit (ri*2 + cj) = query block ri, key block cj
// of the tile).
__host__ __device__ inline int32_t pack_entry(int it, int hl, int sub) {
  return (it & 0xFFFFF) | ((hl & 0xFF) << 20) | ((sub & 0xF) << 28);
}
__host__ __device__ inline int entry_it(int32_t e) { return e & 0xFFFFF; }
__host__ __device__ inline int entry_hl(int32_t e) { return (e >> 20) & 0xFF; }
__host__ __device__ inline int entry_sub(int32_t e) { return (int)(((uint32_t)e) >> 28); }

// Sliding window (preTokens / nextTokens rows of the parameter table; left and
// right window edges as on the FlashAttentionScore page): query s and key t of
// one sequence, both counted from that sequence's first token, pair up iff
// s - pre <= t <= s + next. The host clamps pre and next to +-2^40 (positions
// stay below 2^31, so the clamp changes no pair and int64 never overflows).
constexpr int64_t kWinClamp = int64_t(1) << 40;

// The rectangle of positions [s0, s1) x [t0, t1) (both non-empty) holds at
// least one pair of the window.
__host__ __device__ inline bool win_meets(int64_t s0, int64_t s1, int64_t t0, int64_t t1,
                                          int64_t pre, int64_t next) {
  return t0 - (s1 - 1) <= next && (t1 - 1) - s0 >= -pre;
}
// Every pair of the rectangle lies in the window.
__host__ __device__ inline bool win_covers(int64_t s0, int64_t s1, int64_t t0, int64_t t1,
                                           int64_t pre, int64_t next) {
  return (t1 - 1) - s0 <= next && t0 - (s1 - 1) >= -pre;
}
// Positions x of the other axis with pos + dlo <= x <= pos + dhi, as the
// half-open range [lo, hi) of offsets from `base`, clipped to [0, 128]
// (a query row: dlo = -pre, dhi = next; a key row: dlo = -next, dhi = pre).
__host__ __device__ inline int2 win_span(int64_t pos, int64_t base, int64_t dlo, int64_t dhi) {
  int64_t lo = pos + dlo - base, hi = pos + dhi - base + 1;
  lo = lo < 0 ? 0 : (lo > 128 ? 128 : lo);
  hi = hi < 0 ? 0 : (hi > 128 ? 128 : hi);
  return make_int2((int)lo, (int)hi);
}

// Token mask attenMask (parameter table row attenMaskOptional: the atten_mask
// of S = Mask(scale*Q*K^T, atten_mask); a true entry masks the pair out, as
// on the FlashAttentionScore page): one [maxSq, maxSkv] matrix for every
// batch and head, indexed by per-sequence positions. The preprocess packs it
// into bit rows (query-major and key-major) and classifies each 64x64
// sub-block: 0 every pair masked, 1 some, 2 none (positions outside the
// matrix count as masked; they lie past every sequence length).
constexpr int kAmAll = 0, kAmSome = 1, kAmNone = 2;

// A block (i, j) of bx x by tokens has a pair the token mask keeps.
__host__ __device__ inline bool am_block_meets(const uint8_t* sub, int sk, int i, int j, int bx,
                                               int by) {
  for (int qi = i * bx / 64; qi < (i + 1) * bx / 64; ++qi)
    for (int qj = j * by / 64; qj < (j + 1) * by / 64; ++qj)
      if (sub[qi * sk + qj] != kAmAll) return true;
  return false;
}

// Bits lo .. hi-1 of a 32-bit word (the part of [lo, hi) inside [0, 32)).
__host__ __device__ inline uint32_t bit_range(int lo, int hi) {
  lo = lo < 0 ? 0 : lo;
  hi = hi > 32 ? 32 : hi;
  if (hi <= lo) return 0u;
  const uint32_t below_hi = hi == 32 ? 0xFFFFFFFFu : ((1u << hi) - 1u);
  return below_hi & ~((1u << lo) - 1u);
}

// Everything the kernels need, passed by value.
struct Plan {
  // problem
  int B, N1, N2, G, D;
  int bx, by, rb, cb;      // block shape, blocks per tile
  int Mq, Mk;              // mask dims (blocks); 0 when the mask is null
  int Mq_t, Mk_t;          // max tiles per sequence (query / key)
  int layout, dtype;
  int has_mask;
  int Sq, Skv;             // BNSD padded lengths (TND: longest sequence)
  int Tq, Tkv;             // TND token totals (BNSD: 0)
  float scale, scale_log2; // scale, scale*log2(e)
  // tensors (device)
  const void* q;
  const void* k;
  const void* v;
  const void* dout;
  const void* out;
  const float* lse;
  const uint8_t* mask;
  void* dq;
  void* dk;
  void* dv;
  int64_t mask_sb, mask_sh, mask_si;    // mask strides (b, h, i); j stride 1
  int64_t dq_st[4], dk_st[4], dv_st[4]; // output strides (elements), layout order
  int dq_vec, dkv_vec;                  // outputs allow 16-byte row stores
  int dkv_tma;                          // dK / dV written by TMA stores (BwdMaps dk, dv)
  int det;                              // deterministic dQ: separate query-tile pass, no reduce-adds
  int win;                              // a sliding window cuts some pair of the problem
  int64_t win_pre, win_next;            // its limits (clamped to +-kWinClamp)
  int am;                               // the token mask attenMask applies (maskType 1)
  const uint32_t* am_row;               // [Mq_t*128][am_wk]: bit k of word w = pair (s, 32w+k) masked
  const uint32_t* am_col;               // [Mk_t*128][am_wq]: bit k of word w = pair (32w+k, t) masked
  const uint8_t* am_sub;                // [Mq_t*2][am_sk] class of each 64x64 sub-block
  int am_wk, am_wq, am_sk;              // row strides (words, words, bytes)
  // per-batch info in the workspace (int32 [B] each)
  const int* lq;
  const int* lk;
  const int* cu_q;       // TND token offsets (BNSD: 0)
  const int* cu_k;
  const int* qrow;       // padded query-row offset of batch b (multiple of 128)
  const int* krow;       // padded key-tile offset of batch b (in tiles)
  const int* qtile_b;    // batch of padded query tile r/128
  int Rq;                // padded query rows per head (sum of 128*ceil(lq/128))
  int n_qtiles;          // Rq / 128
  // workspace arrays
  int* header;
  float* lse2;           // [N1][Rq] lse*log2(e) (0 on padding rows)
  float* dvec;           // [N1][Rq] rowsum(dout*out) (0 on padding rows)
  float* dqacc;          // [N1][Rq][D] fp32 dQ accumulator
  int* colcnt;           // [NC] active tiles of grouped column (b,g,jt,hl)
  int* colptr;           // [NC+1]
  int32_t* entries;      // [max_entries]
  int4* items;           // [max_items] {gcol, e_begin, e_end, slot}
  int* colinfo;          // [NGC] -1 empty, -2 single item, >=0 slot
  int* fin_tiles;        // [NGC] key tiles (gc) with colinfo != -2, count in the header
  float* slots;          // [max_slots][2][128][D] fp32 dK, dV partials
  int NC;                // B*N2*Mk_t*G grouped columns
  int NGC;               // B*N2*Mk_t key tiles
  int max_items, max_slots, max_entries;
  int num_sms;
  int min_chunk;         // smallest split chunk
  int n_waves;           // work items are ordered in this many waves of (b, kv head)
  int wait_test;         // test of the bounded waits: 1 = one wait on a barrier nothing completes
};

}  // namespace bsa
