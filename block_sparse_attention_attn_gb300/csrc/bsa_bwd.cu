// bsa_bwd.cu - block-sparse attention backward on the sm_103a tensor cores.
//
// Computes, for every selected (query tile, key tile) pair, the five dense
// contractions of the backward formulas of the aclnnBlockSparseAttentionGrad
// page (section 计算公式):
//     S^T  = K Q^T                 P^T  = exp(scale*S^T - lse)   (recompute)
//     dP^T = V dO^T                dS^T = P^T o (dP^T - D)
//     dV  += P^T dO                dK  += dS^T Q                 (TMEM accumulators)
//     dQ   = dS K                  -> fp32 accumulator in global memory (atomics)
// with D = rowsum(dO o attentionOut) from the preprocess kernel.
//
// Design (one persistent CTA per SM, 512 threads, warp-specialised):
//   warp 12     TMA producer: K/V tiles of the key tile (once per work item),
//               then a 2-stage ring of Q tiles (with their lse/D rows) and
//               one dO buffer.
//   warp 13     tcgen05 MMA issuer for dP, dV and S (one thread) and TMEM
//               owner (512 columns); warp 14 issues dQ and dK.
//   warps 0-7   "softmax" warpgroups: TMEM lane t = key row t; warpgroup w
//               handles query columns [64w, 64w+64): P^T (into TMEM, packed, as
//               the A operand of the dV MMA) and dS (into shared memory, the
//               operand of both the dQ and the dK MMA).
//   warps 8-11  drain: dQ tile TMEM -> registers (the whole row in one load, so
//               the columns go straight back to the next dP) -> fp32
//               accumulator (TMA reduce-add); at the end of a work item, dK/dV
//               TMEM -> output (or fp32 slot for split columns). Warp 15 only
//               lends its registers to the drain warps.
// A work item is one key tile (b, kv head g, jt) with the query tiles of all
// G query heads of the group that select it (so the GQA sum happens in TMEM),
// or a chunk of such a list when the planner split a long column.
//
// MMA order for tile n of an item: dP(n), dV(n), S(n+1), dQ(n), dK(n). S of
// the next tile is issued as soon as dV(n) has read P^T(n) out of the S
// columns, so the softmax warps compute P(n+1) while the tensor pipe runs
// dQ(n) and dK(n); dQ(n) goes first so the drain empties its TMEM columns
// while dK(n) runs.
//
// TMEM columns: [0,128) dV^T, [128,256) dK^T, [256,384) S^T -> P^T,
// [384,512) dP^T, then dQ once the softmax warps have read dP^T.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bsa_common.h"
#include "bsa_launch.h"
#include "bsa_device.cuh"
#include "sm103_ptx.cuh"

namespace bsa {
namespace {

constexpr int kThreads = 512;
constexpr int kProducerWarp = 12;  // warps 12-15: producer, two MMA issuers, one idle warp
constexpr int kMmaWarp = 13;   // dP, dV, S; TMEM owner
constexpr int kMma2Warp = 14;  // dQ, dK
constexpr int kDrainWarp0 = 8;
constexpr int kPanel = 128 * 128;  // 128 rows x 128 bytes (64 x 16-bit), one swizzle span
constexpr int kStages = 2;
constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColP = 384;
// Registers per thread after the hand-over (launch: 512 x 128): the control
// warpgroup gives 48 of its 128 to the drain warpgroup, which reads a whole
// dQ row (D values) out of TMEM at once: 128 + 128 + 176 + 80 = 4 x 128.
// Each budget has its own copy of the out-of-line wait loop (wait tags).
constexpr int kRegsCtl = 80, kRegsDrain = 176;
constexpr int kTagCtl = 1, kTagSoftmax = 2, kTagDrain = 3;

// Offset of K-step k (16 elements) inside a 128-byte-swizzled tile, in the
// 16-byte units of a shared-memory descriptor's address field: K-major tiles
// step 32 bytes within a 64-element panel, MN-major tiles step 16 rows.
__host__ __device__ constexpr uint64_t kmaj_step(int k) {
  return static_cast<uint64_t>(((k >> 2) * kPanel + (k & 3) * 32) >> 4);
}
__host__ __device__ constexpr uint64_t mn_step(int k) { return static_cast<uint64_t>((k * 2048) >> 4); }

enum Bar {
  kBufFull0 = 0, kBufFull1, kBufAux0, kBufAux1, kBufEmpty0, kBufEmpty1,
  kQFull0, kQFull1, kQEmpty0, kQEmpty1, kQAux0, kQAux1,
  kDoFull, kDoEmpty, kDoAux,
  kSFull, kDpFull, kPReady, kDsReady, kDvDone, kDqFull, kDqEmpty, kDsFree,
  kAccFull, kAccEmpty,
  kItemFull0, kItemFull1, kItemEmpty0, kItemEmpty1,
  kDrainBar, kDrainBar2, kNeverBar,
  kNumBars
};

// Shared memory (D = 128: 224 KB of tiles): K, V (per item), Q in a 2-stage
// ring (with its lse/D rows), one dO buffer, the dS tile (operand of the dQ
// and dK MMAs) and a 32 KB dQ staging buffer. The fp32 dQ tile (128 x D) is
// staged in 32 x 32 boxes, 64 columns at a time.
template <int D>
struct Smem {
  static constexpr int kTileBytes = (D / 64) * kPanel;
  static constexpr int oK = 0;
  static constexpr int oV = oK + kTileBytes;
  static constexpr int oQ = oV + kTileBytes;
  static constexpr int odO = oQ + kStages * kTileBytes;
  static constexpr int odS = odO + kTileBytes;
  static constexpr int oStg = odS + 2 * kPanel;
  static constexpr int oLse = oStg + 2 * kPanel;
  static constexpr int oDv = oLse + kStages * 128 * 4;
  static constexpr int oBar = oDv + kStages * 128 * 4;
  static constexpr int oMisc = (oBar + kNumBars * 8 + 63) / 64 * 64;  // int4 slots need 16 B
  static_assert(oMisc % 16 == 0, "misc area must be 16-byte aligned");
  static constexpr int kBytes = oMisc + 64;
};

// Zero rows [r0, 128) of a [128 x 64*panels] swizzled tile (full 128-byte rows,
// so the swizzle does not matter). Executed by one warp.
__device__ __noinline__ void zero_rows(uint8_t* tile, int panels, int r0, int lane) {
  const int nrows = 128 - r0;
  const int n16 = nrows * 8;  // 16-byte chunks per panel
  for (int pnl = 0; pnl < panels; ++pnl) {
    uint4* base = reinterpret_cast<uint4*>(tile + pnl * kPanel + r0 * 128);
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

// S^T = K Q^T for one tile (K-major K and Q tiles), then a commit to `bar`.
// Kept out of line: it is issued from three places in the MMA warp.
template <int D>
__device__ __noinline__ void mma_s_tile(uint32_t d_tmem, uint32_t aK, uint32_t aQ, uint32_t idesc,
                                        uint64_t* bar) {
  const uint64_t dA = sdesc_sw128(aK, 16, 1024), dB = sdesc_sw128(aQ, 16, 1024);
#pragma unroll
  for (int k = 0; k < D / 16; ++k) mma_ss(d_tmem, dA + kmaj_step(k), dB + kmaj_step(k), idesc, k > 0);
  tc_commit(bar);
}

// Packed fp32 pairs (two lanes of one 64-bit register): one instruction for
// two columns of the dS computation.
__device__ __forceinline__ uint64_t f2(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void f2split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Claims the next work item from the device queue (lane 0) and hands it to
// every lane of the warp; x = -1 marks the end of the work.
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

// EM: instantiated with the element-mask code (sliding window, Plan::win, and
// token mask, Plan::am); the plain instance carries none of it.
template <int D, int DT, bool EM>
__global__ void __launch_bounds__(kThreads, 1)
    k_bwd(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
          const __grid_constant__ CUtensorMap tm_acc, const __grid_constant__ CUtensorMap tm_dk,
          const __grid_constant__ CUtensorMap tm_dv, const Plan p) {
  using S = Smem<D>;
  using E = Elem<DT>;
  using T = typename E::T;
  constexpr int kPanels = D / 64;
  constexpr uint32_t kIdS = idesc_f16(128, 128, E::kAB, 0, 0);   // S^T, dP^T
  constexpr uint32_t kIdKV = idesc_f16(128, D, E::kAB, 0, 1);    // dV (A in TMEM), dK
  constexpr uint32_t kIdQ = idesc_f16(128, D, E::kAB, 1, 1);     // dQ

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
    mbar_init(&bars[kBufFull0], 1);   // K/V buffer loaded (TMA bytes, or producer after zeroing)
    mbar_init(&bars[kBufFull1], 1);
    mbar_init(&bars[kBufAux0], 1);    // K/V buffer bytes of a key tile that ends early
    mbar_init(&bars[kBufAux1], 1);
    mbar_init(&bars[kBufEmpty0], 1);  // MMA commit after the buffer's last reader
    mbar_init(&bars[kBufEmpty1], 1);
    mbar_init(&bars[kQFull0], 2);
    mbar_init(&bars[kQFull1], 2);
    mbar_init(&bars[kQEmpty0], 1);  // dK MMA commit (the last reader of Q)
    mbar_init(&bars[kQEmpty1], 1);
    mbar_init(&bars[kQAux0], 1);
    mbar_init(&bars[kQAux1], 1);
    mbar_init(&bars[kDoFull], 1);
    mbar_init(&bars[kDoEmpty], 1);  // dV MMA commit (the last reader of dO)
    mbar_init(&bars[kDoAux], 1);
    mbar_init(&bars[kSFull], 1);
    mbar_init(&bars[kDpFull], 1);
    mbar_init(&bars[kPReady], 8);
    mbar_init(&bars[kDsReady], 8);
    mbar_init(&bars[kDvDone], 1);   // dV MMA commit (P^T read, S columns free)
    mbar_init(&bars[kDqFull], 1);
    mbar_init(&bars[kDqEmpty], 4);
    mbar_init(&bars[kDsFree], 1);  // dK MMA commit (the last reader of the dS tile)
    mbar_init(&bars[kAccFull], 2);   // last dV (MMA warp) and last dK (second MMA warp)
    mbar_init(&bars[kAccEmpty], 4);
    mbar_init(&bars[kItemFull0], 1);
    mbar_init(&bars[kItemFull1], 1);
    mbar_init(&bars[kItemEmpty0], 14);
    mbar_init(&bars[kItemEmpty1], 14);
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
    if (p.dkv_tma) {
      tma_prefetch_desc(&tm_dk);
      tma_prefetch_desc(&tm_dv);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  uint8_t* sK = smem + S::oK;
  uint8_t* sV = smem + S::oV;
  uint8_t* sQ0 = smem + S::oQ;
  uint8_t* sdO = smem + S::odO;
  uint8_t* sdS = smem + S::odS;
  uint8_t* sStg = smem + S::oStg;

  // K and V of a work item live in the two key-tile buffers, with roles that
  // alternate from item to item: item ic keeps K in buffer (ic & 1) and V in
  // the other one. The next item's K is then loaded into the buffer whose V
  // was last read by the current item's final dP, and its V into the buffer
  // whose K was last read by the final dQ, so both loads overlap the end of
  // the current item.
  if (warp >= kProducerWarp) {
  regs_release<kRegsCtl>();  // all four warps of the control warpgroup
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    uint32_t n = 0, fc = 0, ic = 0;  // tiles, ring slots filled, non-empty items
    uint32_t aux_cnt[2] = {0u, 0u}, do_aux_cnt = 0, buf_aux_cnt[2] = {0u, 0u};
    uint32_t last_q_par[2] = {0u, 0u}, last_do_par = 0, last_buf_par[2] = {0u, 0u};
    int pending_q[2] = {0, 0}, pending_q_aux[2] = {0, 0};
    int pending_do = 0, pending_do_aux = 0;
    int pending_buf[2] = {0, 0}, pending_buf_aux[2] = {0, 0};
    bool ok = true;
    // Items are claimed one ahead, so the next key tile's K/V can be
    // prefetched into L2 while the current item runs.
    int4 next = claim_item(p, lane);
    auto kv_coords = [&](const ItemInfo& it, int& c1, int& c2) {
      c1 = p.layout == kLayoutBNSD ? it.jt * 128 : it.g;
      c2 = p.layout == kLayoutBNSD ? it.b * p.N2 + it.g : p.cu_k[it.b] + it.jt * 128;
    };
    // K or V of item `it` into buffer `bi` (free once the previous item's last
    // reader of that buffer completed); a key tile that ends early is loaded
    // through the aux barrier, its rows past the key length are cleared and
    // then the full barrier is released by hand.
    auto load_buf = [&](int bi, const CUtensorMap* tm, const ItemInfo& it, int t_valid) -> bool {
      if (!mbar_wait<kTagCtl>(&bars[kBufEmpty0 + bi], (ic & 1) ^ 1, abort_flag)) {
        record_error(p.header, kErrWaitKV);
        return false;
      }
      const bool tail = t_valid < 128;
      uint8_t* dst = bi == 0 ? sK : sV;
      if (lane == 0) {
        int c1, c2;
        kv_coords(it, c1, c2);
        uint64_t* tb = tail ? &bars[kBufAux0 + bi] : &bars[kBufFull0 + bi];
        mbar_arrive_expect_tx(tb, S::kTileBytes);
        const uint64_t pol = l2_policy_evict_first();  // K/V: read once per item
        for (int pn = 0; pn < kPanels; ++pn)
          tma_load_3d_hint(dst + pn * kPanel, tm, tb, pn * 64, c1, c2, pol);
      }
      last_buf_par[bi] = ic & 1;
      pending_buf[bi] = tail ? 0 : 1;
      pending_buf_aux[bi] = tail ? 1 : 0;
      if (tail) {
        if (!mbar_wait<kTagCtl>(&bars[kBufAux0 + bi], buf_aux_cnt[bi] & 1, abort_flag)) {
          record_error(p.header, kErrWaitKV);
          return false;
        }
        buf_aux_cnt[bi]++;
        pending_buf_aux[bi] = 0;
        zero_rows(dst, kPanels, t_valid, lane);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBufFull0 + bi]);
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
      const int Lq = p.lq[ii.b], Lk = p.lk[ii.b];
      const int t_valid = Lk - ii.jt * 128;
      const int kb = ic & 1;
      for (int e = ii.e0; e < ii.e1 && ok; ++e) {
        if (e == ii.e0 && next.x >= 0 && lane == 0) {
          // the next item's K/V into L2, one item before they are loaded
          const ItemInfo nx = decode_item(p, next);
          if (nx.e0 < nx.e1) {
            int c1, c2;
            kv_coords(nx, c1, c2);
            for (int pn = 0; pn < kPanels; ++pn) {
              tma_prefetch_l2_3d(&tm_k, pn * 64, c1, c2);
              tma_prefetch_l2_3d(&tm_v, pn * 64, c1, c2);
            }
          }
        }
        const int32_t ent = load_entry(p, e);
        const int it = entry_it(ent);
        const int h = ii.g * p.G + entry_hl(ent);
        const int st = n & 1;
        const int q0 = it * 128;
        const bool tail = (Lq - q0) < 128;
        const int c1 = p.layout == kLayoutBNSD ? q0 : h;
        const int c2 = p.layout == kLayoutBNSD ? ii.b * p.N1 + h : p.cu_q[ii.b] + q0;
        // Q (stage st) with its lse / D rows
        if (!mbar_wait<kTagCtl>(&bars[kQEmpty0 + st], ((n >> 1) & 1) ^ 1, abort_flag)) {
          record_error(p.header, kErrWaitQ);
          ok = false;
          break;
        }
        uint8_t* sQ = sQ0 + st * S::kTileBytes;
        if (lane == 0) {
          uint64_t* tb = tail ? &bars[kQAux0 + st] : &bars[kQFull0 + st];
          mbar_arrive_expect_tx(tb, S::kTileBytes);
          for (int pn = 0; pn < kPanels; ++pn) tma_load_3d(sQ + pn * kPanel, &tm_q, tb, pn * 64, c1, c2);
        }
        last_q_par[st] = (n >> 1) & 1;
        pending_q[st] = tail ? 0 : 1;
        pending_q_aux[st] = tail ? 1 : 0;
        {
          const int64_t ro = (int64_t)h * p.Rq + p.qrow[ii.b] + q0 + 4 * lane;
          const float4 l4 = *reinterpret_cast<const float4*>(p.lse2 + ro);
          const float4 d4 = *reinterpret_cast<const float4*>(p.dvec + ro);
          // negated: the softmax warps add it with a packed fp32x2 FMA
          reinterpret_cast<float4*>(sLse + st * 128)[lane] = make_float4(-l4.x, -l4.y, -l4.z, -l4.w);
          reinterpret_cast<float4*>(sDv + st * 128)[lane] = d4;
        }
        __syncwarp();
        if (tail) {
          if (!mbar_wait<kTagCtl>(&bars[kQAux0 + st], aux_cnt[st] & 1, abort_flag)) {
            record_error(p.header, kErrWaitQ);
            ok = false;
            break;
          }
          aux_cnt[st]++;
          pending_q_aux[st] = 0;
          zero_rows(sQ, kPanels, Lq - q0, lane);
          fence_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          mbar_arrive(&bars[kQFull0 + st]);
          if (tail) mbar_arrive(&bars[kQFull0 + st]);
        }
        // K and V of the item: K's buffer is free once the previous item's
        // last dP (which read V from it) completed, V's once its last dQ did
        if (e == ii.e0) {
#pragma unroll 1
          for (int w = 0; w < 2 && ok; ++w) ok = load_buf(kb ^ w, w == 0 ? &tm_k : &tm_v, ii, t_valid);
          if (!ok) break;
        }
        // dO (single buffer): free once the previous tile's dV MMA completed
        if (!mbar_wait<kTagCtl>(&bars[kDoEmpty], (n & 1) ^ 1, abort_flag)) {
          record_error(p.header, kErrWaitQ);
          ok = false;
          break;
        }
        if (lane == 0) {
          uint64_t* tb = tail ? &bars[kDoAux] : &bars[kDoFull];
          mbar_arrive_expect_tx(tb, S::kTileBytes);
          for (int pn = 0; pn < kPanels; ++pn) tma_load_3d(sdO + pn * kPanel, &tm_do, tb, pn * 64, c1, c2);
        }
        last_do_par = n & 1;
        pending_do = tail ? 0 : 1;
        pending_do_aux = tail ? 1 : 0;
        if (tail) {
          if (!mbar_wait<kTagCtl>(&bars[kDoAux], do_aux_cnt & 1, abort_flag)) {
            record_error(p.header, kErrWaitQ);
            ok = false;
            break;
          }
          do_aux_cnt++;
          pending_do_aux = 0;
          zero_rows(sdO, kPanels, Lq - q0, lane);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kDoFull]);
        }
        ++n;
      }
      ++ic;
    }
    if (*abort_flag) {
      // let copies still in flight land before the CTA exits
      for (int st = 0; st < 2; ++st) {
        if (pending_q[st]) mbar_wait_drain(&bars[kQFull0 + st], last_q_par[st]);
        if (pending_q_aux[st]) mbar_wait_drain(&bars[kQAux0 + st], aux_cnt[st] & 1);
        if (pending_buf[st]) mbar_wait_drain(&bars[kBufFull0 + st], last_buf_par[st]);
        if (pending_buf_aux[st]) mbar_wait_drain(&bars[kBufAux0 + st], buf_aux_cnt[st] & 1);
      }
      if (pending_do) mbar_wait_drain(&bars[kDoFull], last_do_par);
      if (pending_do_aux) mbar_wait_drain(&bars[kDoAux], do_aux_cnt & 1);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    uint32_t n = 0, fc = 0, ic = 0;  // tiles, ring slots read, non-empty items
    const uint32_t aBuf0 = smem_u32(sK), aBuf1 = smem_u32(sV);
    const uint32_t adO = smem_u32(sdO);
    int where = 0;
    // next non-empty item from the ring (its entry range [e0, e1)): 1 item,
    // 0 end of work, -1 wait failed
    auto fetch = [&](int& e0, int& e1) -> int {
      while (true) {
        const int slot = fc & 1;
        if (!mbar_wait<kTagCtl>(&bars[kItemFull0 + slot], (fc >> 1) & 1, abort_flag)) return -1;
        const int4 raw = item_slot[slot];
        __syncwarp();
        if (elect_one()) mbar_arrive(&bars[kItemEmpty0 + slot]);
        ++fc;
        if (raw.x < 0) return 0;
        e0 = raw.y;
        e1 = raw.z;
        if (e0 < e1) return 1;
      }
    };
    // S^T(m) = K Q(m)^T into the S columns
    auto issue_s = [&](uint32_t m, uint32_t aK) {
      if (elect_one())
        mma_s_tile<D>(tmem + kColS, aK, smem_u32(sQ0 + (m & 1) * S::kTileBytes), kIdS, &bars[kSFull]);
      __syncwarp();
    };
    int ce0 = 0, ce1 = 0;
    int have = fetch(ce0, ce1);
    if (have < 0) where = kErrWaitItem;
    if (have > 0) {  // S of the very first tile
      // test of the bounded waits: a barrier no one arrives at runs out, the
      // CTA unwinds and the host reads the error code
      if (p.wait_test && !mbar_wait<kTagCtl>(&bars[kNeverBar], 0, abort_flag)) where = kErrWaitTest;
      else if (!mbar_wait<kTagCtl>(&bars[kBufFull0], 0, abort_flag)) where = kErrWaitKV;
      else if (!mbar_wait<kTagCtl>(&bars[kQFull0], 0, abort_flag)) where = kErrWaitQ;
      else {
        tc_fence_after();
        issue_s(0, aBuf0);
      }
    }
    while (have > 0 && !where) {
      const int kb = ic & 1, vb = kb ^ 1;
      const uint32_t aK = kb ? aBuf1 : aBuf0, aV = kb ? aBuf0 : aBuf1;
      int ne0 = 0, ne1 = 0;
      int have_next = 0;
      bool first = true;
      for (int e = ce0; e < ce1; ++e) {
        const bool last = e + 1 == ce1;
        // dP^T = V dO^T: the dP columns hold dQ of the previous tile until
        // the drain warps have read it
        if (!mbar_wait<kTagCtl>(&bars[kDqEmpty], (n & 1) ^ 1, abort_flag)) { where = kErrWaitDQ; break; }
        if (first && !mbar_wait<kTagCtl>(&bars[kBufFull0 + vb], ic & 1, abort_flag)) { where = kErrWaitKV; break; }
        if (!mbar_wait<kTagCtl>(&bars[kDoFull], n & 1, abort_flag)) { where = kErrWaitQ; break; }
        tc_fence_after();
        if (elect_one()) {  // dP^T = V dO^T
          const uint64_t dV = sdesc_sw128(aV, 16, 1024), dO = sdesc_sw128(adO, 16, 1024);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            mma_ss(tmem + kColP, dV + kmaj_step(k), dO + kmaj_step(k), kIdS, k > 0);
          }
          tc_commit(&bars[kDpFull]);
          if (last) tc_commit(&bars[kBufEmpty0 + vb]);  // V read for the last time
        }
        __syncwarp();
        if (!mbar_wait<kTagCtl>(&bars[kPReady], n & 1, abort_flag)) { where = kErrWaitP; break; }
        // the first dV/dK MMAs of an item overwrite the accumulators: the drain
        // warps must have read the previous item's dK/dV
        if (first && !mbar_wait<kTagCtl>(&bars[kAccEmpty], (ic & 1) ^ 1, abort_flag)) { where = kErrWaitAcc; break; }
        tc_fence_after();
        if (elect_one()) {  // dV^T += P^T dO  (A = P^T in TMEM, packed)
          const uint64_t dOmn = sdesc_sw128(adO, kPanel, 1024);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t acol = kColS + 64 * (k >> 2) + 8 * (k & 3);
            mma_ts(tmem + kColDV, tmem + acol, dOmn + mn_step(k), kIdKV, (first && k == 0) ? 0u : 1u);
          }
          tc_commit(&bars[kDoEmpty]);  // dO may be reloaded once dP and dV completed
          tc_commit(&bars[kDvDone]);
          if (last) tc_commit(&bars[kAccFull]);  // dV of the item complete
        }
        __syncwarp();
        // S of the next tile -- after the item's last tile, of the next
        // item, whose K sits in this item's V buffer -- once dV has read P^T
        // out of the S columns
        bool next_s = !last;
        if (last) {
          have_next = fetch(ne0, ne1);
          if (have_next < 0) { where = kErrWaitItem; break; }
          if (have_next > 0) {
            if (p.wait_test && !mbar_wait<kTagCtl>(&bars[kNeverBar], 0, abort_flag)) { where = kErrWaitTest; break; }
            if (!mbar_wait<kTagCtl>(&bars[kBufFull0 + vb], (ic + 1) & 1, abort_flag)) { where = kErrWaitKV; break; }
            next_s = true;
          }
        }
        if (next_s) {
          if (!mbar_wait<kTagCtl>(&bars[kDvDone], n & 1, abort_flag)) { where = kErrWaitMisc; break; }
          if (!mbar_wait<kTagCtl>(&bars[kQFull0 + ((n + 1) & 1)], ((n + 1) >> 1) & 1, abort_flag)) {
            where = kErrWaitQ;
            break;
          }
          tc_fence_after();
          issue_s(n + 1, last ? aV : aK);
        }
        first = false;
        ++n;
      }
      if (where) break;
      ++ic;
      ce0 = ne0;
      ce1 = ne1;
      have = have_next;
    }
    if (where) record_error(p.header, where);
    if (*abort_flag) {  // wait for MMAs still in flight before TMEM is freed
      if (elect_one()) tc_commit(&bars[kDrainBar]);
      __syncwarp();
      mbar_wait_drain(&bars[kDrainBar], 0);
    }
  } else if (warp == kMma2Warp) {
    // ------------------------------------------------ MMA issuer: dQ and dK
    // A second issuing warp keeps the tensor pipe fed while the first one
    // waits for P, dO or the S columns, and vice versa. The two share no
    // barrier phase: dQ and dK follow dS, which the softmax warps signal only
    // after the S and dP MMAs of the tile have completed.
    uint32_t n = 0, itc = 0, ic = 0;  // tiles, ring slots read, non-empty items
    const uint32_t aBuf0 = smem_u32(sK), aBuf1 = smem_u32(sV), adS = smem_u32(sdS);
    int where = 0;
    while (true) {
      const int slot = itc & 1;
      if (!mbar_wait<kTagCtl>(&bars[kItemFull0 + slot], (itc >> 1) & 1, abort_flag)) { where = kErrWaitItem; break; }
      const int4 raw = item_slot[slot];
      __syncwarp();
      if (elect_one()) mbar_arrive(&bars[kItemEmpty0 + slot]);
      ++itc;
      if (raw.x < 0) break;
      const int e0 = raw.y, e1 = raw.z;
      if (e0 >= e1) continue;
      const int kb = ic & 1;
      const uint32_t aK = kb ? aBuf1 : aBuf0;
      for (int e = e0; e < e1; ++e) {
        const bool first = e == e0, last = e + 1 == e1;
        const int st = n & 1;
        const uint32_t aQ = smem_u32(sQ0 + st * S::kTileBytes);
        // with two 64-key blocks per tile, dS is zero on the keys of an
        // unselected block: the dQ product skips their K-steps (keys 16k ..
        // 16k + 15 for step k)
        int kq0 = 0, kq1 = 8;
        if (p.cb == 2) {
          const int sub = entry_sub(load_entry(p, e));
          const bool h0 = ((sub | (sub >> 2)) & 1) != 0, h1 = ((sub | (sub >> 2)) & 2) != 0;
          if (h0 != h1) {
            kq0 = h0 ? 0 : 4;
            kq1 = h0 ? 4 : 8;
          }
        }
        if (!mbar_wait<kTagCtl>(&bars[kDsReady], n & 1, abort_flag)) { where = kErrWaitDS; break; }
        if (first) {  // this item's K, and dK of the previous item read out
          if (!mbar_wait<kTagCtl>(&bars[kBufFull0 + kb], ic & 1, abort_flag)) { where = kErrWaitKV; break; }
          if (!mbar_wait<kTagCtl>(&bars[kAccEmpty], (ic & 1) ^ 1, abort_flag)) { where = kErrWaitAcc; break; }
        }
        tc_fence_after();
        if (elect_one()) {
          // dQ = dS K  (A = dS, MN-major; B = K, MN-major) into the dP columns,
          // which the softmax warps have read before they signalled dS (not in
          // the deterministic mode, where a separate pass computes dQ)
          const uint64_t dSmn = sdesc_sw128(adS, kPanel, 1024), dKmn = sdesc_sw128(aK, kPanel, 1024);
          const uint64_t dSk = sdesc_sw128(adS, 16, 1024), dQmn = sdesc_sw128(aQ, kPanel, 1024);
          if (!p.det) {
#pragma unroll 1
            for (int k = kq0; k < kq1; ++k) {
              mma_ss(tmem + kColP, dSmn + mn_step(k), dKmn + mn_step(k), kIdQ, k > kq0);
            }
          }
          tc_commit(&bars[kDqFull]);
          if (last) tc_commit(&bars[kBufEmpty0 + kb]);  // K read for the last time
          // dK^T += dS^T Q  (A = dS^T, K-major: the same shared-memory tile)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            mma_ss(tmem + kColDK, dSk + kmaj_step(k), dQmn + mn_step(k), kIdKV,
                   (first && k == 0) ? 0u : 1u);
          }
          tc_commit(&bars[kQEmpty0 + st]);
          tc_commit(&bars[kDsFree]);
          if (last) tc_commit(&bars[kAccFull]);  // dK of the item complete
        }
        __syncwarp();
        ++n;
      }
      if (where) break;
      ++ic;
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
    const int wg = warp >> 2;  // query columns [64 wg, 64 wg + 64)
    const int qd = warp & 3;   // TMEM lane quadrant
    const int t = qd * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    uint32_t n = 0, itc = 0;
    int where = 0;
    while (true) {
      const int slot = itc & 1;
      if (!mbar_wait<kTagSoftmax>(&bars[kItemFull0 + slot], (itc >> 1) & 1, abort_flag)) { where = kErrWaitItem; break; }
      const int4 raw = item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + slot]);
      if (raw.x < 0) break;
      const ItemInfo ii = decode_item(p, raw);
      if (ii.e0 >= ii.e1) { ++itc; continue; }
      const int Lk = p.lk[ii.b];
      const bool t_ok = (ii.jt * 128 + t) < Lk;
      // the next tile's entry, and (token mask) its sub-block classes and this
      // thread's mask words, are loaded one tile ahead: each depends on the
      // one before, and they would otherwise stall the start of every tile
      int32_t ent_n = load_entry(p, ii.e0);
      uint32_t cls01_n = 0, cls23_n = 0;  // class bytes of the tile's 2x2 sub-blocks
      uint2 amw_n = make_uint2(0u, 0u);
      auto am_prefetch = [&](int32_t en) {
        const int itn = entry_it(en);
        const uint8_t* sc = p.am_sub + (int64_t)(2 * itn) * p.am_sk + 2 * ii.jt;
        cls01_n = *reinterpret_cast<const uint16_t*>(sc);
        cls23_n = *reinterpret_cast<const uint16_t*>(sc + p.am_sk);
        amw_n = *reinterpret_cast<const uint2*>(p.am_col + ((int64_t)ii.jt * 128 + t) * p.am_wq +
                                                4 * itn + 2 * wg);
      };
      if (EM && p.am) am_prefetch(ent_n);
      for (int e = ii.e0; e < ii.e1; ++e) {
        const int32_t ent = ent_n;
        const uint32_t cls01 = cls01_n, cls23 = cls23_n;
        const uint2 amw = amw_n;
        if (e + 1 < ii.e1) ent_n = load_entry(p, e + 1);
        const int sub = entry_sub(ent);
        const int s_sub = (p.rb == 2) ? wg : 0;
        const int t_sub = (p.cb == 2) ? (t >> 6) : 0;
        // key row t of this thread takes part (inside the key length, in a
        // selected sub-block); query columns past the query length need no
        // test: their lse rows hold +inf, so P is exactly 0 there
        const uint32_t rmask = (t_ok && ((sub >> (s_sub * 2 + t_sub)) & 1)) ? 0xFFFFFFFFu : 0u;
        // element masks: when the sliding window or the token mask cuts this
        // tile (the same answer for the whole CTA), wm0 / wm1 flag the live
        // query columns of this thread's two 32-column chunks
        bool wcut = false;
        uint32_t wm0 = 0xFFFFFFFFu, wm1 = 0xFFFFFFFFu;
        if (EM) {
          const int it = entry_it(ent);
          const int64_t s0 = (int64_t)it * 128, t0 = (int64_t)ii.jt * 128;
          if (p.win && !win_covers(s0, s0 + 128, t0, t0 + 128, p.win_pre, p.win_next)) {
            wcut = true;
            const int2 w = win_span(t0 + t, s0 + 64 * wg, -p.win_next, p.win_pre);
            wm0 = bit_range(w.x, w.y);
            wm1 = bit_range(w.x - 32, w.y - 32);
          }
          if (p.am) {
            const uint32_t c = cls01 & cls23;
            if (((c & 0xFFu) & (c >> 8)) != (uint32_t)kAmNone) {  // some sub-block has a masked pair
              wcut = true;
              wm0 &= ~amw.x;
              wm1 &= ~amw.y;
            }
          }
        }
        const int st = n & 1;
        if (!mbar_wait<kTagSoftmax>(&bars[kQFull0 + st], (n >> 1) & 1, abort_flag)) { where = kErrWaitQ; break; }
        if (!mbar_wait<kTagSoftmax>(&bars[kSFull], n & 1, abort_flag)) { where = kErrWaitS; break; }
        tc_fence_after();
        const float* nlse2 = sLse + st * 128;  // -lse2 of the tile's query columns
        const float* dv = sDv + st * 128;
        // P^T of this thread's 64 columns, packed to the operand type (the
        // same rounded values feed the dV MMA and dS = P o (dP - D))
        uint32_t Ppk[32];
        {
          uint32_t x[64];  // both 32-column chunks in one TMEM load
          tmem_ld64(tmem + lane_off + kColS + 64 * wg, x);
          const uint64_t c2 = f2(__float_as_uint(p.scale_log2), __float_as_uint(p.scale_log2));
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int s0 = 64 * wg + 32 * c;
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const float4 l4 = reinterpret_cast<const float4*>(nlse2 + s0)[j4];
              const int xi = 32 * c + 4 * j4;
              float t0, t1, t2, t3;
              f2split(fma2(f2(x[xi], x[xi + 1]), c2, f2(__float_as_uint(l4.x), __float_as_uint(l4.y))), t0, t1);
              f2split(fma2(f2(x[xi + 2], x[xi + 3]), c2, f2(__float_as_uint(l4.z), __float_as_uint(l4.w))), t2, t3);
              const float p0 = ex2_approx(t0);
              const float p1 = ex2_approx(t1);
              const float p2 = ex2_approx(t2);
              const float p3 = ex2_approx(t3);
              Ppk[16 * c + 2 * j4] = E::pack(p0, p1) & rmask;
              Ppk[16 * c + 2 * j4 + 1] = E::pack(p2, p3) & rmask;
            }
            if (wcut) {  // word j holds columns 2j (low half) and 2j + 1 (high half)
              const uint32_t wm = c ? wm1 : wm0;
#pragma unroll
              for (int j = 0; j < 16; ++j)
                Ppk[16 * c + j] &= ((wm >> (2 * j)) & 1u ? 0x0000FFFFu : 0u) |
                                   ((wm >> (2 * j + 1)) & 1u ? 0xFFFF0000u : 0u);
            }
          }
          // packed P^T over the first half of this warpgroup's S columns
          tmem_st32(tmem + lane_off + kColS + 64 * wg, Ppk);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kPReady]);
        if (EM && p.am && e + 1 < ii.e1) am_prefetch(ent_n);  // ent_n has arrived by now
        if (!mbar_wait<kTagSoftmax>(&bars[kDpFull], n & 1, abort_flag)) { where = kErrWaitDP; break; }
        if (!mbar_wait<kTagSoftmax>(&bars[kDsFree], (n & 1) ^ 1, abort_flag)) { where = kErrWaitMisc; break; }
        tc_fence_after();
        {
          uint32_t y[64];  // dP of both 32-column chunks in one TMEM load
          tmem_ld64(tmem + lane_off + kColP + 64 * wg, y);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int s0 = 64 * wg + 32 * c;
            uint32_t pk[16];
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const float4 d4 = reinterpret_cast<const float4*>(dv + s0)[j4];
              const int yi = 32 * c + 4 * j4;
              const float2 p01 = E::unpack(Ppk[16 * c + 2 * j4]);
              const float2 p23 = E::unpack(Ppk[16 * c + 2 * j4 + 1]);
              // two columns per packed fp32x2 subtract and multiply
              float a0, a1, b0, b1;
              f2split(mul2(sub2(f2(y[yi], y[yi + 1]), f2(__float_as_uint(d4.x), __float_as_uint(d4.y))),
                           f2(__float_as_uint(p01.x), __float_as_uint(p01.y))), a0, a1);
              f2split(mul2(sub2(f2(y[yi + 2], y[yi + 3]), f2(__float_as_uint(d4.z), __float_as_uint(d4.w))),
                           f2(__float_as_uint(p23.x), __float_as_uint(p23.y))), b0, b1);
              pk[2 * j4] = E::pack(a0, a1);
              pk[2 * j4 + 1] = E::pack(b0, b1);
            }
            // dS into shared memory: panel wg, row t, 16-byte chunk cc holds
            // s = 64 wg + 8 cc .. +7, swizzled by t & 7 -- the MN-major A
            // operand (M = query s) of the dQ MMA and the K-major A operand
            // (M = key t) of the dK MMA.
            uint8_t* rowp = sdS + wg * kPanel + t * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int cc = 4 * c + q;
              *reinterpret_cast<uint4*>(rowp + ((cc ^ (t & 7)) << 4)) =
                  make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
          }
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kDsReady]);
        ++n;
      }
      if (where) break;
      ++itc;
    }
    if (where) record_error(p.header, where);
  } else {
    regs_claim<kRegsDrain>();
    // -------------------------------------------------------------- drain
    const int qd = warp & 3;
    const int r = qd * 32 + lane;  // TMEM lane: query row (dQ) / key row (dK, dV)
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    uint32_t n = 0, itc = 0, ic = 0;  // tiles, ring slots read, non-empty items
    int where = 0;
    while (true) {
      const int slot = itc & 1;
      if (!mbar_wait<kTagDrain>(&bars[kItemFull0 + slot], (itc >> 1) & 1, abort_flag)) { where = kErrWaitItem; break; }
      const int4 raw = item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + slot]);
      if (raw.x < 0) break;
      const ItemInfo ii = decode_item(p, raw);
      if (ii.e0 >= ii.e1) { ++itc; continue; }
      const int Lk = p.lk[ii.b];
      for (int e = ii.e0; e < ii.e1; ++e) {
        const int32_t ent = load_entry(p, e);
        const int it = entry_it(ent);
        const int h = ii.g * p.G + entry_hl(ent);
        if (!mbar_wait<kTagDrain>(&bars[kDqFull], n & 1, abort_flag)) { where = kErrWaitDQ; break; }
        tc_fence_after();
        if (p.det) {  // no dQ here: the columns go straight back to the next dP
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kDqEmpty]);
          ++n;
          continue;
        }
        // dQ tile -> fp32 accumulator with TMA reduce-adds. The thread's whole
        // row (D columns) comes out of TMEM in one load, so the columns go
        // back to the next dP before any staging. Each warp owns 32 rows and
        // an 8 KB part of the staging buffer: two 32 x 32 fp32 boxes
        // (128-byte swizzled), i.e. 64 columns at a time. Rows past the query
        // length carry exact zeros (dS = 0 there) and land in the padded part
        // of the accumulator.
        const int grow = h * p.Rq + p.qrow[ii.b] + it * 128 + qd * 32;
        uint8_t* boxes = sStg + qd * 8192;
        uint8_t* rowp = boxes + lane * 128;
        uint32_t acc[D];
        if constexpr (D == 128) tmem_ld128(tmem + lane_off + kColP, acc);
        else tmem_ld64(tmem + lane_off + kColP, acc);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kDqEmpty]);  // TMEM columns free for the next dP
        const uint64_t pol = l2_policy_evict_last();   // keep dQ accumulator rows in L2
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf) {
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
      // dK / dV of the key tile
      if (!mbar_wait<kTagDrain>(&bars[kAccFull], ic & 1, abort_flag)) { where = kErrWaitAcc; break; }
      tc_fence_after();
      const int trow = ii.jt * 128 + r;
      const bool row_ok = (p.layout == kLayoutBNSD) ? (trow < p.Skv) : (trow < Lk);
      int64_t ok_off = 0, ov_off = 0;
      int64_t sdk = 1, sdv = 1;
      if (p.layout == kLayoutBNSD) {
        ok_off = ii.b * p.dk_st[0] + ii.g * p.dk_st[1] + (int64_t)trow * p.dk_st[2];
        ov_off = ii.b * p.dv_st[0] + ii.g * p.dv_st[1] + (int64_t)trow * p.dv_st[2];
        sdk = p.dk_st[3];
        sdv = p.dv_st[3];
      } else {
        ok_off = ((int64_t)p.cu_k[ii.b] + trow) * p.dk_st[0] + ii.g * p.dk_st[1];
        ov_off = ((int64_t)p.cu_k[ii.b] + trow) * p.dv_st[0] + ii.g * p.dv_st[1];
        sdk = p.dk_st[2];
        sdv = p.dv_st[2];
      }
      float* slot_base = ii.slot >= 0 ? p.slots + (int64_t)ii.slot * 2 * 128 * D : nullptr;
      // Whole tiles go out through the staging buffer as TMA stores: each warp
      // packs its 32 rows into 32 x 64 boxes (128-byte swizzled) and stores
      // them; a TND tile that ends inside the sequence, split columns (fp32
      // slots) and outputs without a store view take the per-row path.
      const bool tma_out = p.dkv_tma && slot_base == nullptr &&
                           (p.layout == kLayoutBNSD || ii.jt * 128 + 128 <= Lk);
      if (tma_out) {
        // The accumulator rows leave TMEM before any TMA store: dK is read,
        // scaled, packed and staged, then dV is read and packed, and the
        // columns go back to the next item's first dV / dK; the stores follow.
        uint8_t* boxes = sStg + qd * 8192;
        const int trow0 = ii.jt * 128 + qd * 32;
        uint8_t* wk = boxes;
        uint8_t* wv = (D == 64) ? boxes + 4096 : boxes;
        // packed row words (16 per 32 columns) -> 128-byte-swizzled 32 x 64 boxes
        auto stage = [&](const uint32_t (&w)[D / 2], uint8_t* wb) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint8_t* rowp = wb + (c >> 1) * 4096 + lane * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(rowp + ((((c & 1) * 4 + q) ^ (lane & 7)) << 4)) =
                  make_uint4(w[16 * c + 4 * q], w[16 * c + 4 * q + 1], w[16 * c + 4 * q + 2],
                             w[16 * c + 4 * q + 3]);
          }
          fence_async_smem();
          __syncwarp();
        };
        auto store = [&](uint8_t* wb, const CUtensorMap* tm) {
          if (lane == 0) {
#pragma unroll
            for (int bx = 0; bx < D / 64; ++bx) {
              if (p.layout == kLayoutBNSD)
                tma_store_4d(tm, wb + bx * 4096, bx * 64, trow0, ii.g, ii.b);
              else
                tma_store_3d(tm, wb + bx * 4096, bx * 64, ii.g, p.cu_k[ii.b] + trow0);
            }
            bulk_commit_group();
          }
        };
        {
          uint32_t kp[D / 2];
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf) {
            uint32_t x[64];
            tmem_ld64(tmem + lane_off + kColDK + 64 * hf, x);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              kp[32 * hf + j] = E::pack(__uint_as_float(x[2 * j]) * p.scale,
                                        __uint_as_float(x[2 * j + 1]) * p.scale);
          }
          if (lane == 0) bulk_wait_read_all();  // dQ boxes of the last tile were read
          __syncwarp();
          stage(kp, wk);
        }
        uint32_t vp[D / 2];
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf) {
          uint32_t x[64];
          tmem_ld64(tmem + lane_off + kColDV + 64 * hf, x);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            vp[32 * hf + j] = E::pack(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kAccEmpty]);  // TMEM dK / dV free
        store(wk, &tm_dk);
        if (D == 128) {  // the dK boxes must be read before dV reuses them
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
        }
        stage(vp, wv);
        store(wv, &tm_dv);
      } else {  // rare: kept compact (not unrolled)
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
          const uint32_t col = which == 0 ? kColDK : kColDV;
          const float mul = which == 0 ? p.scale : 1.f;
          T* out = static_cast<T*>(which == 0 ? p.dk : p.dv) + (which == 0 ? ok_off : ov_off);
          const int64_t sd = which == 0 ? sdk : sdv;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t x[32];
            tmem_ld32(tmem + lane_off + col + 32 * c, x);
            if (slot_base != nullptr) {
              if (r < Lk - ii.jt * 128) {
                float4* d4 = reinterpret_cast<float4*>(slot_base + (which * 128 + r) * D + 32 * c);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  atomicAdd(d4 + j, make_float4(__uint_as_float(x[4 * j]) * mul,
                                                __uint_as_float(x[4 * j + 1]) * mul,
                                                __uint_as_float(x[4 * j + 2]) * mul,
                                                __uint_as_float(x[4 * j + 3]) * mul));
              }
            } else if (row_ok) {
              if (p.dkv_vec) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  uint4 u;
                  u.x = E::pack(__uint_as_float(x[8 * j]) * mul, __uint_as_float(x[8 * j + 1]) * mul);
                  u.y = E::pack(__uint_as_float(x[8 * j + 2]) * mul, __uint_as_float(x[8 * j + 3]) * mul);
                  u.z = E::pack(__uint_as_float(x[8 * j + 4]) * mul, __uint_as_float(x[8 * j + 5]) * mul);
                  u.w = E::pack(__uint_as_float(x[8 * j + 6]) * mul, __uint_as_float(x[8 * j + 7]) * mul);
                  *reinterpret_cast<uint4*>(out + 32 * c + 8 * j) = u;
                }
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  const uint32_t pk = E::pack(__uint_as_float(x[j]) * mul, 0.f);
                  out[(32 * c + j) * sd] = *reinterpret_cast<const T*>(&pk);
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kAccEmpty]);
      }
      ++itc;
      ++ic;
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

template <int D, int DT, bool EM>
cudaError_t launch_t(const Plan& p, const BwdMaps& m, cudaStream_t st) {
  const size_t smem = Smem<D>::kBytes;
  // The register hand-over only balances when every thread starts with 128
  // registers (the claim would otherwise wait for registers nobody frees).
  static const int regs = [] {
    cudaFuncAttributes fa{};
    return cudaFuncGetAttributes(&fa, k_bwd<D, DT, EM>) == cudaSuccess ? fa.numRegs : -1;
  }();
  static_assert(2 * 128 + kRegsDrain + kRegsCtl == 4 * 128, "register hand-over must balance");
  if (regs != 128) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(k_bwd<D, DT, EM>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int grid = p.num_sms;
  if (p.max_items < grid) grid = p.max_items;
  if (grid < 1) grid = 1;
  k_bwd<D, DT, EM><<<grid, kThreads, smem, st>>>(m.q, m.k, m.v, m.dout, m.dqacc, m.dk, m.dv, p);
  return cudaGetLastError();
}

template <bool EM>
cudaError_t launch_w(const Plan& p, const BwdMaps& m, cudaStream_t st) {
  if (p.dtype == kDtBF16)
    return p.D == 128 ? launch_t<128, kDtBF16, EM>(p, m, st) : launch_t<64, kDtBF16, EM>(p, m, st);
  return p.D == 128 ? launch_t<128, kDtF16, EM>(p, m, st) : launch_t<64, kDtF16, EM>(p, m, st);
}

}  // namespace

size_t bwd_smem_bytes(int D) { return D == 128 ? Smem<128>::kBytes : Smem<64>::kBytes; }

cudaError_t launch_bwd(const Plan& p, const BwdMaps& m, cudaStream_t st) {
  return (p.win || p.am) ? launch_w<true>(p, m, st) : launch_w<false>(p, m, st);
}

}  // namespace bsa
