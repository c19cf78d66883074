// bsa_bwd_k64.cu - block-sparse attention backward for key blocks of 64
// tokens (blockShape [bx, 64], head dim 128) on the sm_103a tensor cores.
//
// The same five contractions per selected block as k_bwd (the backward
// formulas of the aclnnBlockSparseAttentionGrad page, section 计算公式), but
// laid out query-major, so that a single 64-key block is a full-rate MMA
// (M = 128 queries or 128 head dimensions, N = 64 keys) instead of half of a
// 128-key tile whose other half is multiplied and masked away:
//     S      = Q K_h^T    (M = 128 queries, N = 64 keys, K = D)
//     P      = exp(scale*S - lse)             dP = dO V_h^T
//     dS     = P o (dP - D)
//     dV_h^T += dO^T P    (M = D head dims, N = 64 keys, K = 128 queries)
//     dK_h^T += Q^T dS                         (TMEM accumulators)
//     dQ      = dS K_h    (M = 128 queries, N = D, K = 64 keys)
//                          -> fp32 accumulator in global memory (TMA reduce-add)
// A work item is the one k_bwd uses: a 128-key tile (key blocks 2jt and
// 2jt + 1) of one kv head, with the query tiles of all G heads of the group
// that select a block of it. The kernel makes two passes over the item's list,
// one per key block h: a pass keeps K_h and V_h (64 rows each) in shared
// memory and dV_h^T, dK_h^T in TMEM, and visits only the query tiles whose
// sub-block mask selects block h, so an unselected block is never loaded or
// multiplied.
//
// Roles (one persistent CTA per SM, 512 threads):
//   warp 12     TMA producer: K_h / V_h at the start of a pass, Q (with its
//               lse / D rows) and dO in 2-stage rings, one stage per visit.
//   warp 13     MMA issuer for S and dP (two TMEM buffers each) and TMEM owner.
//   warp 14     MMA issuer for dV, dK and dQ.
//   warps 0-7   softmax: thread = query row (TMEM lane), warpgroup w = keys
//               [32w, 32w + 32) of the block; P and dS go to shared memory as
//               [query][key] tiles, the operand of the dV, dK and dQ MMAs.
//   warps 8-11  drain: dQ -> fp32 accumulator after every visit; at the end of
//               a pass dK_h, dV_h (thread = head dim) -> output rows, or into
//               an fp32 slot when the planner split the column.
//   warp 15     lends its registers to the drain warps.
//
// TMEM columns: [0,64) dV_h^T, [64,128) dK_h^T, [128,256) dQ, [256,384) S
// (two 64-column buffers), [384,512) dP (two buffers).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bsa_common.h"
#include "bsa_launch.h"
#include "bsa_device.cuh"
#include "sm103_ptx.cuh"

namespace bsa {
namespace {

constexpr int kThreads = 512;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;   // S, dP; TMEM owner
constexpr int kMma2Warp = 14;  // dV, dK, dQ
constexpr int kDrainWarp0 = 8;
constexpr int kD = 128;
constexpr int kPanel = 128 * 128;        // 128 rows x 128 bytes: Q, dO, P, dS
constexpr int kPanelH = 64 * 128;        // 64 rows x 128 bytes: K_h, V_h
constexpr int kTileBytes = 2 * kPanel;   // 128 x D 16-bit
constexpr int kHalfBytes = 2 * kPanelH;  // 64 x D 16-bit
constexpr uint32_t kColDV = 0, kColDK = 64, kColQ = 128, kColS = 256, kColP = 384;
// Register budgets after the hand-over (launch: 512 x 128), as in k_bwd: the
// drain warpgroup reads a whole dQ row (128 columns) out of TMEM at once.
constexpr int kRegsCtl = 80, kRegsDrain = 176;
constexpr int kTagCtl = 1, kTagSoftmax = 2, kTagDrain = 3;

// K-step k (16 elements) of a K-major 128-byte-swizzled operand, in the
// 16-byte units of a descriptor's address field: 32 bytes within a
// 64-element panel, `panel` bytes on to the next panel.
__host__ __device__ constexpr uint64_t kstep(int k, int panel) {
  return static_cast<uint64_t>(((k >> 2) * panel + (k & 3) * 32) >> 4);
}
// K-step k of an MN-major operand: 16 rows of 128 bytes.
__host__ __device__ constexpr uint64_t mstep(int k) { return static_cast<uint64_t>((k * 2048) >> 4); }

enum Bar {
  kBufFull0 = 0, kBufFull1, kBufAux0, kBufAux1, kBufEmpty0, kBufEmpty1,
  kQFull0, kQFull1, kQEmpty0, kQEmpty1, kQAux0, kQAux1,
  kDoFull0, kDoFull1, kDoEmpty0, kDoEmpty1, kDoAux0, kDoAux1,
  kSFull0, kSFull1, kSFree0, kSFree1, kDpFull0, kDpFull1, kDpFree0, kDpFree1,
  kPReady, kPFree, kDsReady, kDsFree,
  kDqFull, kDqEmpty, kAccFull, kAccEmpty,
  kItemFull0, kItemFull1, kItemEmpty0, kItemEmpty1,
  kDrainBar, kDrainBar2, kNeverBar,
  kNumBars
};

// Shared memory (226 KB): two 16 KB key-block buffers (K_h and V_h, roles
// alternating from pass to pass), Q and dO in 2-stage rings, the P and dS
// tiles ([128 queries][64 keys], one swizzle panel each), a 32 KB dQ staging
// buffer, the lse / D rows of both Q stages, barriers.
struct Smem {
  static constexpr int oB0 = 0;
  static constexpr int oB1 = oB0 + kHalfBytes;
  static constexpr int oQ = oB1 + kHalfBytes;
  static constexpr int odO = oQ + 2 * kTileBytes;
  static constexpr int oP = odO + 2 * kTileBytes;
  static constexpr int odS = oP + kPanel;
  static constexpr int oStg = odS + kPanel;
  static constexpr int oLse = oStg + 2 * kPanel;
  static constexpr int oDv = oLse + 2 * 128 * 4;
  static constexpr int oBar = oDv + 2 * 128 * 4;
  static constexpr int oMisc = (oBar + kNumBars * 8 + 63) / 64 * 64;
  static constexpr int kBytes = oMisc + 64;
};
static_assert(Smem::kBytes <= 227 * 1024, "shared memory budget");

// Zero rows [r0, rows) of a [rows x 128] 16-bit tile stored as two swizzled
// panels `panel` bytes apart (whole 128-byte rows, so the swizzle does not
// matter). Executed by one warp.
__device__ __noinline__ void zero_rows(uint8_t* tile, int rows, int panel, int r0, int lane) {
  if (r0 < 0) r0 = 0;
  const int n16 = (rows - r0) * 8;
  for (int pnl = 0; pnl < 2; ++pnl) {
    uint4* base = reinterpret_cast<uint4*>(tile + pnl * panel + r0 * 128);
    for (int i = lane; i < n16; i += 32) base[i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

struct ItemInfo {
  int b, g, jt, e0, e1, slot;
};

__device__ __forceinline__ ItemInfo decode_item(const Plan& p, int4 it) {
  ItemInfo r;
  r.jt = it.x % p.Mk_t;
  const int bg = it.x / p.Mk_t;
  r.g = bg % p.N2;
  r.b = bg / p.N2;
  r.e0 = it.y;
  r.e1 = it.z;
  r.slot = it.w;
  return r;
}

// Next work item from the device queue (lane 0), handed to the whole warp;
// x = -1 marks the end of the work.
__device__ __forceinline__ int4 claim_item(const Plan& p, int lane) {
  int4 it = make_int4(-1, 0, 0, -1);
  if (lane == 0) {
    const int idx = atomicAdd(&p.header[kHdrWorkCounter], 1);
    if (idx < p.header[kHdrNumItems]) it = checked_item(p, p.items[idx]);
  }
  it.x = __shfl_sync(0xffffffffu, it.x, 0);
  it.y = __shfl_sync(0xffffffffu, it.y, 0);
  it.z = __shfl_sync(0xffffffffu, it.z, 0);
  it.w = __shfl_sync(0xffffffffu, it.w, 0);
  return it;
}

// Contiguous global -> shared bulk copy (addresses 16-byte aligned, size a
// multiple of 16), completion counted as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// First entry at or after e (before e1) whose sub-block mask selects key
// block h of the tile in either query block.
__device__ __forceinline__ int next_visit(const Plan& p, int e, int e1, int h) {
  while (e < e1) {
    const int sub = entry_sub(load_entry(p, e));
    if ((((sub | (sub >> 2)) >> h) & 1) != 0) break;
    ++e;
  }
  return e;
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 1)
    k_bwd_k64(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_acc, const Plan p) {
  using S = Smem;
  using E = Elem<DT>;
  using T = typename E::T;
  constexpr uint32_t kIdS = idesc_f16(128, 64, E::kAB, 0, 0);   // S, dP
  constexpr uint32_t kIdKV = idesc_f16(128, 64, E::kAB, 1, 1);  // dV^T, dK^T
  constexpr uint32_t kIdQ = idesc_f16(128, kD, E::kAB, 0, 1);   // dQ

  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::oBar);
  int* misc = reinterpret_cast<int*>(smem + S::oMisc);
  volatile int* abort_flag = misc + 0;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 1);
  int4* item_slot = reinterpret_cast<int4*>(misc + 4);  // [2], 16-byte aligned
  float* sLse = reinterpret_cast<float*>(smem + S::oLse);
  float* sDv = reinterpret_cast<float*>(smem + S::oDv);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if ((smem_u32(smem) & 1023u) != 0) {  // tiles need 1024-byte alignment
    if (threadIdx.x == 0) record_error(p.header, kErrSmemAlign);
    return;
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kBufFull0 + i], 1);   // TMA bytes, or the producer after zeroing a tail
      mbar_init(&bars[kBufAux0 + i], 1);    // bytes of a key block that ends early
      mbar_init(&bars[kBufEmpty0 + i], 1);  // MMA commit after the buffer's last reader
      mbar_init(&bars[kQFull0 + i], 1);     // Q tile + lse / D rows (TMA and bulk-copy bytes)
      mbar_init(&bars[kQEmpty0 + i], 1);    // dK MMA commit
      mbar_init(&bars[kQAux0 + i], 1);
      mbar_init(&bars[kDoFull0 + i], 1);
      mbar_init(&bars[kDoEmpty0 + i], 1);   // commit after the visit's dK / dQ (dV read dO before)
      mbar_init(&bars[kDoAux0 + i], 1);
      mbar_init(&bars[kSFull0 + i], 1);
      mbar_init(&bars[kSFree0 + i], 8);     // softmax warps have read S
      mbar_init(&bars[kDpFull0 + i], 1);
      mbar_init(&bars[kDpFree0 + i], 8);
      mbar_init(&bars[kItemFull0 + i], 1);
      mbar_init(&bars[kItemEmpty0 + i], 14);
    }
    mbar_init(&bars[kPReady], 8);
    mbar_init(&bars[kPFree], 1);    // dV MMA commit
    mbar_init(&bars[kDsReady], 8);
    mbar_init(&bars[kDsFree], 1);   // dK / dQ MMA commit
    mbar_init(&bars[kDqFull], 1);
    mbar_init(&bars[kDqEmpty], 4);
    mbar_init(&bars[kAccFull], 1);  // last dV / dK of a pass
    mbar_init(&bars[kAccEmpty], 4);
    mbar_init(&bars[kDrainBar], 1);
    mbar_init(&bars[kDrainBar2], 1);
    mbar_init(&bars[kNeverBar], 1);  // nothing arrives here (wait_test)
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_acc);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  uint8_t* sB0 = smem + S::oB0;
  uint8_t* sB1 = smem + S::oB1;
  uint8_t* sQ0 = smem + S::oQ;
  uint8_t* sdO0 = smem + S::odO;
  uint8_t* sP = smem + S::oP;
  uint8_t* sdS = smem + S::odS;
  uint8_t* sStg = smem + S::oStg;

  // Pass pc (counted over the passes that visit something) keeps K_h in
  // buffer (pc & 1) and V_h in the other one: the next pass's K goes into the
  // buffer whose V was last read by the current pass's final dP, its V into
  // the one whose K was last read by the final dQ.
  if (warp >= kProducerWarp) {
  regs_release<kRegsCtl>();  // all four warps of the control warpgroup
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    uint32_t n = 0, fc = 0, pc = 0;  // visits, ring slots filled, passes
    uint32_t q_aux[2] = {0u, 0u}, do_aux[2] = {0u, 0u}, b_aux[2] = {0u, 0u};
    // copies that may still be in flight if the CTA unwinds: the barrier that
    // tracks each stage's last copy (-1 none) and its phase parity
    int pend_q[2] = {-1, -1}, pend_do[2] = {-1, -1}, pend_b[2] = {-1, -1};
    uint32_t par_q[2] = {0u, 0u}, par_do[2] = {0u, 0u}, par_b[2] = {0u, 0u};
    bool ok = true;
    int4 next = claim_item(p, lane);
    auto kv_coords = [&](const ItemInfo& it, int h, int& c1, int& c2) {
      const int t0 = it.jt * 128 + 64 * h;
      c1 = p.layout == kLayoutBNSD ? t0 : it.g;
      c2 = p.layout == kLayoutBNSD ? it.b * p.N2 + it.g : p.cu_k[it.b] + t0;
    };
    // One 16-bit [rows x 128] tile (2 panels) by TMA into dst; a tile with
    // fewer than `rows` live rows goes through the aux barrier, its dead rows
    // are cleared and then `full` is released by hand.
    auto load_tile = [&](uint8_t* dst, int rows, int panel, const CUtensorMap* tm, int c1, int c2,
                         int live, int full, int aux, uint32_t& aux_cnt, int& pend, uint32_t& par,
                         uint32_t full_par, bool once) -> bool {
      const bool tail = live < rows;
      if (lane == 0) {
        uint64_t* tb = tail ? &bars[aux] : &bars[full];
        mbar_arrive_expect_tx(tb, 2 * panel);
        if (once) {  // K / V: read once per pass
          const uint64_t pol = l2_policy_evict_first();
          for (int pn = 0; pn < 2; ++pn) tma_load_3d_hint(dst + pn * panel, tm, tb, pn * 64, c1, c2, pol);
        } else {
          for (int pn = 0; pn < 2; ++pn) tma_load_3d(dst + pn * panel, tm, tb, pn * 64, c1, c2);
        }
      }
      pend = tail ? aux : full;
      par = tail ? (aux_cnt & 1) : full_par;
      if (tail) {
        if (!mbar_wait<kTagCtl>(&bars[aux], aux_cnt & 1, abort_flag)) return false;
        aux_cnt++;
        pend = -1;
        zero_rows(dst, rows, panel, live, lane);
        fence_async_smem();
        __syncwarp();
      }
      return true;
    };
    while (ok) {
      const int4 raw = next;
      const int slot = fc & 1;
      if (!mbar_wait<kTagCtl>(&bars[kItemEmpty0 + slot], ((fc >> 1) & 1) ^ 1, abort_flag)) {
        record_error(p.header, kErrWaitItem);
        break;
      }
      if (lane == 0) {
        item_slot[slot] = raw;
        mbar_arrive(&bars[kItemFull0 + slot]);
      }
      ++fc;
      if (raw.x < 0) break;
      next = claim_item(p, lane);
      const ItemInfo ii = decode_item(p, raw);
      if (ii.e0 >= ii.e1) continue;
      if (next.x >= 0 && lane == 0) {  // the next item's K / V into L2
        const ItemInfo nx = decode_item(p, next);
        if (nx.e0 < nx.e1) {
          for (int h = 0; h < 2; ++h) {
            int c1, c2;
            kv_coords(nx, h, c1, c2);
            for (int pn = 0; pn < 2; ++pn) {
              tma_prefetch_l2_3d(&tm_k, pn * 64, c1, c2);
              tma_prefetch_l2_3d(&tm_v, pn * 64, c1, c2);
            }
          }
        }
      }
      const int Lq = p.lq[ii.b], Lk = p.lk[ii.b];
      for (int hb = 0; hb < 2 && ok; ++hb) {
        const int kb = pc & 1;
        const int t_live = Lk - (ii.jt * 128 + 64 * hb);
        bool first = true;
        for (int e = next_visit(p, ii.e0, ii.e1, hb); e < ii.e1; e = next_visit(p, e + 1, ii.e1, hb)) {
          const int32_t ent = load_entry(p, e);
          const int h = ii.g * p.G + entry_hl(ent);
          const int st = n & 1;
          const uint32_t ph = (n >> 1) & 1;
          const int q0 = entry_it(ent) * 128;
          const int c1 = p.layout == kLayoutBNSD ? q0 : h;
          const int c2 = p.layout == kLayoutBNSD ? ii.b * p.N1 + h : p.cu_q[ii.b] + q0;
          // Q (stage st) with its lse / D rows, all asynchronous: the
          // producer never waits on a global load
          if (!mbar_wait<kTagCtl>(&bars[kQEmpty0 + st], ph ^ 1, abort_flag)) {
            record_error(p.header, kErrWaitQ);
            ok = false;
            break;
          }
          {
            uint8_t* sQ = sQ0 + st * kTileBytes;
            const bool qtail = Lq - q0 < 128;
            const int qb = qtail ? kQAux0 + st : kQFull0 + st;
            if (lane == 0) {
              const int64_t ro = (int64_t)h * p.Rq + p.qrow[ii.b] + q0;
              mbar_arrive_expect_tx(&bars[qb], kTileBytes + 2 * 128 * 4);
              for (int pn = 0; pn < 2; ++pn) tma_load_3d(sQ + pn * kPanel, &tm_q, &bars[qb], pn * 64, c1, c2);
              bulk_load(sLse + st * 128, p.lse2 + ro, 128 * 4, &bars[qb]);
              bulk_load(sDv + st * 128, p.dvec + ro, 128 * 4, &bars[qb]);
            }
            pend_q[st] = qb;
            par_q[st] = qtail ? (q_aux[st] & 1) : ph;
            if (qtail) {  // rows past the query length cleared, then released by hand
              if (!mbar_wait<kTagCtl>(&bars[qb], q_aux[st] & 1, abort_flag)) {
                record_error(p.header, kErrWaitQ);
                ok = false;
                break;
              }
              q_aux[st]++;
              pend_q[st] = -1;
              zero_rows(sQ, 128, kPanel, Lq - q0, lane);
              fence_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bars[kQFull0 + st]);
            }
          }
          // K_h and V_h of the pass
          if (first) {
            for (int w = 0; w < 2 && ok; ++w) {
              const int bi = kb ^ w;
              if (!mbar_wait<kTagCtl>(&bars[kBufEmpty0 + bi], (pc & 1) ^ 1, abort_flag)) {
                record_error(p.header, kErrWaitKV);
                ok = false;
                break;
              }
              int k1, k2;
              kv_coords(ii, hb, k1, k2);
              if (!load_tile(bi ? sB1 : sB0, 64, kPanelH, w == 0 ? &tm_k : &tm_v, k1, k2, t_live,
                             kBufFull0 + bi, kBufAux0 + bi, b_aux[bi], pend_b[bi], par_b[bi], pc & 1,
                             true)) {
                record_error(p.header, kErrWaitKV);
                ok = false;
                break;
              }
              if (t_live < 64 && lane == 0) mbar_arrive(&bars[kBufFull0 + bi]);
            }
            if (!ok) break;
            first = false;
          }
          // dO (stage st): free once the visit's dK / dQ (and so its dV) completed
          if (!mbar_wait<kTagCtl>(&bars[kDoEmpty0 + st], ph ^ 1, abort_flag)) {
            record_error(p.header, kErrWaitQ);
            ok = false;
            break;
          }
          if (!load_tile(sdO0 + st * kTileBytes, 128, kPanel, &tm_do, c1, c2, Lq - q0, kDoFull0 + st,
                         kDoAux0 + st, do_aux[st], pend_do[st], par_do[st], ph, false)) {
            record_error(p.header, kErrWaitQ);
            ok = false;
            break;
          }
          if (Lq - q0 < 128 && lane == 0) mbar_arrive(&bars[kDoFull0 + st]);
          ++n;
        }
        if (!first) ++pc;
      }
    }
    if (*abort_flag) {  // let copies still in flight land before the CTA exits
      for (int st = 0; st < 2; ++st) {
        if (pend_q[st] >= 0) mbar_wait_drain(&bars[pend_q[st]], par_q[st]);
        if (pend_do[st] >= 0) mbar_wait_drain(&bars[pend_do[st]], par_do[st]);
        if (pend_b[st] >= 0) mbar_wait_drain(&bars[pend_b[st]], par_b[st]);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------- MMA issuer: S and dP
    uint32_t n = 0, itc = 0, pc = 0;
    const uint32_t aB0 = smem_u32(sB0), aB1 = smem_u32(sB1);
    int where = 0;
    bool tested = false;
    while (!where) {
      const int slot = itc & 1;
      if (!mbar_wait<kTagCtl>(&bars[kItemFull0 + slot], (itc >> 1) & 1, abort_flag)) { where = kErrWaitItem; break; }
      const int4 raw = item_slot[slot];
      __syncwarp();
      if (elect_one()) mbar_arrive(&bars[kItemEmpty0 + slot]);
      __syncwarp();
      ++itc;
      if (raw.x < 0) break;
      const int e0 = raw.y, e1 = raw.z;
      for (int hb = 0; hb < 2 && e0 < e1 && !where; ++hb) {
        const int kb = pc & 1;
        const uint32_t aK = kb ? aB1 : aB0, aV = kb ? aB0 : aB1;
        bool first = true;
        for (int e = next_visit(p, e0, e1, hb); e < e1;) {
          const int en = next_visit(p, e + 1, e1, hb);
          const bool last = en >= e1;
          const int st = n & 1, bf = n & 1;
          const uint32_t ph = (n >> 1) & 1;
          // test of the bounded waits: a barrier no one arrives at runs out,
          // the CTA unwinds and the host reads the error code
          if (p.wait_test && !tested) {
            tested = true;
            if (!mbar_wait<kTagCtl>(&bars[kNeverBar], 0, abort_flag)) { where = kErrWaitTest; break; }
          }
          if (!mbar_wait<kTagCtl>(&bars[kSFree0 + bf], ph ^ 1, abort_flag)) { where = kErrWaitS; break; }
          if (first && !mbar_wait<kTagCtl>(&bars[kBufFull0 + kb], pc & 1, abort_flag)) { where = kErrWaitKV; break; }
          if (!mbar_wait<kTagCtl>(&bars[kQFull0 + st], ph, abort_flag)) { where = kErrWaitQ; break; }
          tc_fence_after();
          if (elect_one()) {  // S = Q K_h^T
            const uint64_t dA = sdesc_sw128(smem_u32(sQ0 + st * kTileBytes), 16, 1024);
            const uint64_t dB = sdesc_sw128(aK, 16, 1024);
#pragma unroll
            for (int k = 0; k < kD / 16; ++k)
              mma_ss(tmem + kColS + 64 * bf, dA + kstep(k, kPanel), dB + kstep(k, kPanelH), kIdS, k > 0);
            tc_commit(&bars[kSFull0 + bf]);
          }
          __syncwarp();
          if (!mbar_wait<kTagCtl>(&bars[kDpFree0 + bf], ph ^ 1, abort_flag)) { where = kErrWaitDP; break; }
          if (first && !mbar_wait<kTagCtl>(&bars[kBufFull0 + (kb ^ 1)], pc & 1, abort_flag)) { where = kErrWaitKV; break; }
          if (!mbar_wait<kTagCtl>(&bars[kDoFull0 + st], ph, abort_flag)) { where = kErrWaitQ; break; }
          tc_fence_after();
          if (elect_one()) {  // dP = dO V_h^T
            const uint64_t dA = sdesc_sw128(smem_u32(sdO0 + st * kTileBytes), 16, 1024);
            const uint64_t dB = sdesc_sw128(aV, 16, 1024);
#pragma unroll
            for (int k = 0; k < kD / 16; ++k)
              mma_ss(tmem + kColP + 64 * bf, dA + kstep(k, kPanel), dB + kstep(k, kPanelH), kIdS, k > 0);
            tc_commit(&bars[kDpFull0 + bf]);
            if (last) tc_commit(&bars[kBufEmpty0 + (kb ^ 1)]);  // V_h read for the last time
          }
          __syncwarp();
          first = false;
          ++n;
          e = en;
        }
        if (!first) ++pc;
      }
    }
    if (where) record_error(p.header, where);
    if (*abort_flag) {  // wait for MMAs still in flight before TMEM is freed
      if (elect_one()) tc_commit(&bars[kDrainBar]);
      __syncwarp();
      mbar_wait_drain(&bars[kDrainBar], 0);
    }
  } else if (warp == kMma2Warp) {
    // -------------------------------------------- MMA issuer: dV, dK and dQ
    uint32_t n = 0, itc = 0, pc = 0;
    const uint32_t aB0 = smem_u32(sB0), aB1 = smem_u32(sB1);
    const uint32_t aP = smem_u32(sP), adS = smem_u32(sdS);
    int where = 0;
    while (!where) {
      const int slot = itc & 1;
      if (!mbar_wait<kTagCtl>(&bars[kItemFull0 + slot], (itc >> 1) & 1, abort_flag)) { where = kErrWaitItem; break; }
      const int4 raw = item_slot[slot];
      __syncwarp();
      if (elect_one()) mbar_arrive(&bars[kItemEmpty0 + slot]);
      __syncwarp();
      ++itc;
      if (raw.x < 0) break;
      const int e0 = raw.y, e1 = raw.z;
      for (int hb = 0; hb < 2 && e0 < e1 && !where; ++hb) {
        const int kb = pc & 1;
        const uint32_t aK = kb ? aB1 : aB0;
        bool first = true;
        for (int e = next_visit(p, e0, e1, hb); e < e1;) {
          const int en = next_visit(p, e + 1, e1, hb);
          const bool last = en >= e1;
          const int st = n & 1;
          const uint32_t ph = (n >> 1) & 1;
          if (!mbar_wait<kTagCtl>(&bars[kPReady], n & 1, abort_flag)) { where = kErrWaitP; break; }
          // the first dV / dK of a pass overwrite the accumulators: the drain
          // warps must have read the previous pass's dK / dV
          if (first && !mbar_wait<kTagCtl>(&bars[kAccEmpty], (pc & 1) ^ 1, abort_flag)) { where = kErrWaitAcc; break; }
          if (!mbar_wait<kTagCtl>(&bars[kDoFull0 + st], ph, abort_flag)) { where = kErrWaitQ; break; }
          tc_fence_after();
          if (elect_one()) {  // dV_h^T += dO^T P  (both MN-major)
            const uint64_t dA = sdesc_sw128(smem_u32(sdO0 + st * kTileBytes), kPanel, 1024);
            const uint64_t dB = sdesc_sw128(aP, kPanel, 1024);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ss(tmem + kColDV, dA + mstep(k), dB + mstep(k), kIdKV, (first && k == 0) ? 0u : 1u);
            tc_commit(&bars[kPFree]);
          }
          __syncwarp();
          if (!mbar_wait<kTagCtl>(&bars[kDsReady], n & 1, abort_flag)) { where = kErrWaitDS; break; }
          if (first && !mbar_wait<kTagCtl>(&bars[kBufFull0 + kb], pc & 1, abort_flag)) { where = kErrWaitKV; break; }
          if (!mbar_wait<kTagCtl>(&bars[kQFull0 + st], ph, abort_flag)) { where = kErrWaitQ; break; }
          // dQ of the previous visit read out of TMEM (not in the
          // deterministic mode, where a separate pass computes dQ)
          if (!p.det && !mbar_wait<kTagCtl>(&bars[kDqEmpty], (n & 1) ^ 1, abort_flag)) { where = kErrWaitDQ; break; }
          tc_fence_after();
          if (elect_one()) {
            // dK_h^T += Q^T dS  (both MN-major)
            const uint64_t dA = sdesc_sw128(smem_u32(sQ0 + st * kTileBytes), kPanel, 1024);
            const uint64_t dB = sdesc_sw128(adS, kPanel, 1024);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ss(tmem + kColDK, dA + mstep(k), dB + mstep(k), kIdKV, (first && k == 0) ? 0u : 1u);
            if (!p.det) {  // dQ = dS K_h  (A = dS K-major, B = K_h MN-major)
              const uint64_t dS = sdesc_sw128(adS, 16, 1024);
              const uint64_t dK = sdesc_sw128(aK, kPanelH, 1024);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_ss(tmem + kColQ, dS + kstep(k, kPanel), dK + mstep(k), kIdQ, k > 0);
              tc_commit(&bars[kDqFull]);
            }
            tc_commit(&bars[kDsFree]);
            tc_commit(&bars[kQEmpty0 + st]);
            tc_commit(&bars[kDoEmpty0 + st]);
            if (last) {
              tc_commit(&bars[kBufEmpty0 + kb]);  // K_h read for the last time
              tc_commit(&bars[kAccFull]);         // dK_h / dV_h of the pass complete
            }
          }
          __syncwarp();
          first = false;
          ++n;
          e = en;
        }
        if (!first) ++pc;
      }
    }
    if (where) record_error(p.header, where);
    if (*abort_flag) {  // wait for this warp's MMAs still in flight
      if (elect_one()) tc_commit(&bars[kDrainBar2]);
      __syncwarp();
      mbar_wait_drain(&bars[kDrainBar2], 0);
    }
  }
  } else if (warp < kDrainWarp0) {
    // ------------------------------------------------------------- softmax
    const int wg = warp >> 2;  // keys [32 wg, 32 wg + 32) of the block
    const int qd = warp & 3;   // TMEM lane quadrant
    const int q = qd * 32 + lane;  // query row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    const uint32_t wcol = 32 * wg;
    uint32_t n = 0, itc = 0;
    int where = 0;
    while (!where) {
      const int slot = itc & 1;
      if (!mbar_wait<kTagSoftmax>(&bars[kItemFull0 + slot], (itc >> 1) & 1, abort_flag)) { where = kErrWaitItem; break; }
      const int4 raw = item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + slot]);
      ++itc;
      if (raw.x < 0) break;
      const ItemInfo ii = decode_item(p, raw);
      const int Lk = p.lk[ii.b];
      for (int hb = 0; hb < 2 && ii.e0 < ii.e1 && !where; ++hb) {
        // keys of this thread's 32 columns inside the key length
        const int kv = Lk - (ii.jt * 128 + 64 * hb + 32 * wg);
        const uint32_t kmask = kv >= 32 ? 0xFFFFFFFFu : (kv <= 0 ? 0u : ((1u << kv) - 1u));
        for (int e = next_visit(p, ii.e0, ii.e1, hb); e < ii.e1; e = next_visit(p, e + 1, ii.e1, hb)) {
          // live keys of the thread's query row: inside the key length and in
          // a selected sub-block (with two query blocks per tile, the row's own
          // block decides); rows past the query length need no test, their
          // lse rows hold +inf, so P is exactly 0 there
          const int sub = entry_sub(load_entry(p, e));
          const bool row_sel = p.rb == 2 ? (((sub >> ((q >> 6) * 2 + hb)) & 1) != 0) : true;
          const uint32_t cm = row_sel ? kmask : 0u;
          const int st = n & 1, bf = n & 1;
          const uint32_t ph = (n >> 1) & 1;
          if (!mbar_wait<kTagSoftmax>(&bars[kQFull0 + st], ph, abort_flag)) { where = kErrWaitQ; break; }
          const float l2 = sLse[st * 128 + q];
          const float dvq = sDv[st * 128 + q];
          if (!mbar_wait<kTagSoftmax>(&bars[kSFull0 + bf], ph, abort_flag)) { where = kErrWaitS; break; }
          tc_fence_after();
          uint32_t x[32];
          tmem_ld32(tmem + lane_off + kColS + 64 * bf + wcol, x);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kSFree0 + bf]);  // S buffer free for the visit after next
          // P of the 32 keys, packed to the operand type (the same rounded
          // values feed the dV MMA and dS = P o (dP - D))
          uint32_t pp[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float p0 = ex2_approx(fmaf(__uint_as_float(x[2 * j]), p.scale_log2, -l2));
            const float p1 = ex2_approx(fmaf(__uint_as_float(x[2 * j + 1]), p.scale_log2, -l2));
            pp[j] = E::pack(p0, p1);
          }
          if (cm != 0xFFFFFFFFu) {  // word j holds keys 2j (low half) and 2j + 1 (high half)
#pragma unroll
            for (int j = 0; j < 16; ++j)
              pp[j] &= ((cm >> (2 * j)) & 1u ? 0x0000FFFFu : 0u) | ((cm >> (2 * j + 1)) & 1u ? 0xFFFF0000u : 0u);
          }
          // P row q into its [query][key] tile: 16-byte chunk c of the row
          // holds keys 8c .. 8c + 7, swizzled by q & 7 (128-byte swizzle)
          if (!mbar_wait<kTagSoftmax>(&bars[kPFree], (n & 1) ^ 1, abort_flag)) { where = kErrWaitMisc; break; }
          {
            uint8_t* rowp = sP + q * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<uint4*>(rowp + (((4 * wg + c) ^ (q & 7)) << 4)) =
                  make_uint4(pp[4 * c], pp[4 * c + 1], pp[4 * c + 2], pp[4 * c + 3]);
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kPReady]);
          if (!mbar_wait<kTagSoftmax>(&bars[kDpFull0 + bf], ph, abort_flag)) { where = kErrWaitDP; break; }
          tc_fence_after();
          uint32_t y[32];
          tmem_ld32(tmem + lane_off + kColP + 64 * bf + wcol, y);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kDpFree0 + bf]);
          uint32_t dd[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 pf = E::unpack(pp[j]);
            dd[j] = E::pack(pf.x * (__uint_as_float(y[2 * j]) - dvq),
                            pf.y * (__uint_as_float(y[2 * j + 1]) - dvq));
          }
          if (!mbar_wait<kTagSoftmax>(&bars[kDsFree], (n & 1) ^ 1, abort_flag)) { where = kErrWaitMisc; break; }
          {
            uint8_t* rowp = sdS + q * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<uint4*>(rowp + (((4 * wg + c) ^ (q & 7)) << 4)) =
                  make_uint4(dd[4 * c], dd[4 * c + 1], dd[4 * c + 2], dd[4 * c + 3]);
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kDsReady]);
          ++n;
        }
      }
    }
    if (where) record_error(p.header, where);
  } else {
    regs_claim<kRegsDrain>();
    // -------------------------------------------------------------- drain
    const int qd = warp & 3;
    const int r = qd * 32 + lane;  // TMEM lane: query row (dQ) / head dim (dK^T, dV^T)
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    uint32_t n = 0, itc = 0, pc = 0;
    int where = 0;
    while (!where) {
      const int slot = itc & 1;
      if (!mbar_wait<kTagDrain>(&bars[kItemFull0 + slot], (itc >> 1) & 1, abort_flag)) { where = kErrWaitItem; break; }
      const int4 raw = item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + slot]);
      ++itc;
      if (raw.x < 0) break;
      const ItemInfo ii = decode_item(p, raw);
      if (ii.e0 >= ii.e1) continue;
      const int Lk = p.lk[ii.b];
      float* slot_base = ii.slot >= 0 ? p.slots + (int64_t)ii.slot * 2 * 128 * kD : nullptr;
      for (int hb = 0; hb < 2 && !where; ++hb) {
        bool any = false;
        for (int e = next_visit(p, ii.e0, ii.e1, hb); e < ii.e1; e = next_visit(p, e + 1, ii.e1, hb)) {
          any = true;
          if (p.det) {  // no dQ here
            ++n;
            continue;
          }
          const int32_t ent = load_entry(p, e);
          const int h = ii.g * p.G + entry_hl(ent);
          if (!mbar_wait<kTagDrain>(&bars[kDqFull], n & 1, abort_flag)) { where = kErrWaitDQ; break; }
          tc_fence_after();
          // dQ of the visit -> fp32 accumulator with TMA reduce-adds: the
          // thread's whole row comes out of TMEM in one load, the columns go
          // back to the next dQ before any staging; each warp owns 32 rows
          // and an 8 KB part of the staging buffer (two 32 x 32 fp32 boxes,
          // 128-byte swizzled), 64 columns at a time. Rows past the query
          // length carry exact zeros and land in the padded accumulator rows.
          const int grow = h * p.Rq + p.qrow[ii.b] + entry_it(ent) * 128 + qd * 32;
          uint8_t* boxes = sStg + qd * 8192;
          uint8_t* rowp = boxes + lane * 128;
          uint32_t acc[kD];
          tmem_ld128(tmem + lane_off + kColQ, acc);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kDqEmpty]);
          const uint64_t pol = l2_policy_evict_last();  // keep dQ accumulator rows in L2
#pragma unroll
          for (int hf = 0; hf < kD / 64; ++hf) {
            if (lane == 0) bulk_wait_read_all();  // the boxes' previous contents were read
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int x0 = 64 * hf + 32 * c + 4 * j;
                *reinterpret_cast<uint4*>(rowp + c * 4096 + ((j ^ (lane & 7)) << 4)) =
                    make_uint4(acc[x0], acc[x0 + 1], acc[x0 + 2], acc[x0 + 3]);
              }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_2d_hint(&tm_acc, boxes, 64 * hf, grow, pol);
              tma_reduce_add_2d_hint(&tm_acc, boxes + 4096, 64 * hf + 32, grow, pol);
              bulk_commit_group();
            }
          }
          __syncwarp();
          ++n;
        }
        if (where) break;
        if (!any && slot_base != nullptr) continue;  // nothing to add to the slot
        // dK_h / dV_h: thread = head dim r, TMEM column = key k of the block
        uint32_t xk[64], xv[64];
        if (any) {
          if (!mbar_wait<kTagDrain>(&bars[kAccFull], pc & 1, abort_flag)) { where = kErrWaitAcc; break; }
          tc_fence_after();
          tmem_ld64(tmem + lane_off + kColDK, xk);
          tmem_ld64(tmem + lane_off + kColDV, xv);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kAccEmpty]);  // TMEM free for the next pass
          ++pc;
        } else {  // no query visits this block: its rows of the tile are zero
#pragma unroll
          for (int k = 0; k < 64; ++k) xk[k] = xv[k] = 0u;
        }
        const int r0 = ii.jt * 128 + 64 * hb;  // first key row of the block
        // (loops fully unrolled: xk / xv stay in registers)
        if (slot_base != nullptr) {
#pragma unroll
          for (int k = 0; k < 64; ++k) {
            if (r0 + k >= Lk) break;
            atomicAdd(slot_base + (64 * hb + k) * kD + r, __uint_as_float(xk[k]) * p.scale);
            atomicAdd(slot_base + (128 + 64 * hb + k) * kD + r, __uint_as_float(xv[k]));
          }
          continue;
        }
        const int rows = p.layout == kLayoutBNSD ? p.Skv - r0 : Lk - r0;  // rows of the output
        int64_t k_off, v_off, k_rs, v_rs, k_cs, v_cs;  // first row, row and column strides
        if (p.layout == kLayoutBNSD) {
          k_off = ii.b * p.dk_st[0] + ii.g * p.dk_st[1] + (int64_t)r0 * p.dk_st[2];
          v_off = ii.b * p.dv_st[0] + ii.g * p.dv_st[1] + (int64_t)r0 * p.dv_st[2];
          k_rs = p.dk_st[2]; v_rs = p.dv_st[2]; k_cs = p.dk_st[3]; v_cs = p.dv_st[3];
        } else {
          k_off = ((int64_t)p.cu_k[ii.b] + r0) * p.dk_st[0] + ii.g * p.dk_st[1];
          v_off = ((int64_t)p.cu_k[ii.b] + r0) * p.dv_st[0] + ii.g * p.dv_st[1];
          k_rs = p.dk_st[0]; v_rs = p.dv_st[0]; k_cs = p.dk_st[2]; v_cs = p.dv_st[2];
        }
        T* outk = static_cast<T*>(p.dk) + k_off;
        T* outv = static_cast<T*>(p.dv) + v_off;
        if (p.dkv_vec) {
          // Unit column stride, 16-byte aligned rows: lanes 2i and 2i + 1
          // swap halves so that each writes one 32-bit word (head dims 2i,
          // 2i + 1) of key 2k2 (even lane) or 2k2 + 1 (odd lane).
          const bool odd = lane & 1;
          const int col = r & ~1;
#pragma unroll
          for (int k2 = 0; k2 < 32; ++k2) {
            const int k = 2 * k2 + (odd ? 1 : 0);
            const uint32_t wk = E::pack(__uint_as_float(xk[2 * k2]) * p.scale,
                                        __uint_as_float(xk[2 * k2 + 1]) * p.scale);
            const uint32_t wv = E::pack(__uint_as_float(xv[2 * k2]), __uint_as_float(xv[2 * k2 + 1]));
            const uint32_t ok = __shfl_xor_sync(0xffffffffu, wk, 1);
            const uint32_t ov = __shfl_xor_sync(0xffffffffu, wv, 1);
            const uint32_t sk = odd ? __byte_perm(ok, wk, 0x7632) : __byte_perm(wk, ok, 0x5410);
            const uint32_t sv = odd ? __byte_perm(ov, wv, 0x7632) : __byte_perm(wv, ov, 0x5410);
            if (k < rows) {
              *reinterpret_cast<uint32_t*>(outk + k * k_rs + col) = sk;
              *reinterpret_cast<uint32_t*>(outv + k * v_rs + col) = sv;
            }
          }
        } else {
#pragma unroll
          for (int k = 0; k < 64; ++k) {
            if (k >= rows) break;
            const uint32_t wk = E::pack(__uint_as_float(xk[k]) * p.scale, 0.f);
            const uint32_t wv = E::pack(__uint_as_float(xv[k]), 0.f);
            outk[k * k_rs + r * k_cs] = *reinterpret_cast<const T*>(&wk);
            outv[k * v_rs + r * v_cs] = *reinterpret_cast<const T*>(&wv);
          }
        }
      }
    }
    if (where) record_error(p.header, where);
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DT>
cudaError_t launch_t(const Plan& p, const BwdMaps& m, cudaStream_t st) {
  const size_t smem = Smem::kBytes;
  // The register hand-over only balances when every thread starts with 128
  // registers (the claim would otherwise wait for registers nobody frees).
  static const int regs = [] {
    cudaFuncAttributes fa{};
    return cudaFuncGetAttributes(&fa, k_bwd_k64<DT>) == cudaSuccess ? fa.numRegs : -1;
  }();
  static_assert(2 * 128 + kRegsDrain + kRegsCtl == 4 * 128, "register hand-over must balance");
  if (regs != 128) return cudaErrorInvalidConfiguration;
  cudaError_t e =
      cudaFuncSetAttribute(k_bwd_k64<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int grid = p.num_sms;
  if (p.max_items < grid) grid = p.max_items;
  if (grid < 1) grid = 1;
  k_bwd_k64<DT><<<grid, kThreads, smem, st>>>(m.q, m.k64, m.v64, m.dout, m.dqacc, p);
  return cudaGetLastError();
}

}  // namespace

bool bwd_k64_applies(const Plan& p) { return p.D == kD && p.by == 64 && !p.win && !p.am; }

cudaError_t launch_bwd_k64(const Plan& p, const BwdMaps& m, cudaStream_t st) {
  if (!bwd_k64_applies(p)) return cudaErrorInvalidValue;
  return p.dtype == kDtBF16 ? launch_t<kDtBF16>(p, m, st) : launch_t<kDtF16>(p, m, st);
}

}  // namespace bsa
