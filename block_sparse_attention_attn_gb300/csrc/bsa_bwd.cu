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
// Design (one persistent CTA per SM, 448 threads, warp-specialised):
//   warp 12     TMA producer: K/V tiles of the key tile (once per work item),
//               then a 2-stage ring of Q/dO tiles plus their lse/D rows.
//   warp 13     tcgen05 MMA issuer (one thread) and TMEM owner (512 columns).
//   warps 0-7   "softmax" warpgroups: TMEM lane t = key row t; warpgroup w
//               handles query columns [64w, 64w+64): P^T (into TMEM, packed, as
//               the A operand of the dV MMA), dS^T (into TMEM for the dK MMA
//               and into shared memory for the dQ MMA).
//   warps 8-11  drain: dQ tile TMEM -> fp32 atomics; at the end of a work
//               item, dK/dV TMEM -> output (or fp32 slot for split columns).
// A work item is one key tile (b, kv head g, jt) with the query tiles of all
// G query heads of the group that select it (so the GQA sum happens in TMEM),
// or a chunk of such a list when the planner split a long column.
//
// TMEM columns: [0,128) dV^T, [128,256) dK^T, [256,384) S^T -> P^T,
// [384,512) dP^T -> dS^T, later reused for dQ.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bsa_common.h"
#include "bsa_launch.h"
#include "sm103_ptx.cuh"

namespace bsa {
namespace {

constexpr int kThreads = 448;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kDrainWarp0 = 8;
constexpr int kPanel = 128 * 128;  // 128 rows x 128 bytes (64 x 16-bit), one swizzle span
constexpr int kStages = 2;
constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColP = 384;

enum Bar {
  kKvTma = 0, kKvFull, kKvEmpty,
  kQFull0, kQFull1, kQEmpty0, kQEmpty1, kQAux0, kQAux1,
  kDoFull, kDoEmpty, kDoAux,
  kSFull, kDpFull, kPReady, kDsReady, kDkDone, kDqFull, kDqEmpty, kDsFree,
  kAccFull, kAccEmpty,
  kItemFull0, kItemFull1, kItemEmpty0, kItemEmpty1,
  kDrainBar, kNeverBar,
  kNumBars
};

// Shared memory (D = 128: 224 KB of tiles): K, V (per item), Q in a 2-stage
// ring (with its lse/D rows), one dO buffer, the dS tile (A operand of the dQ
// MMA) and a 32 KB dQ staging buffer. The fp32 dQ tile (128 x D) is staged in
// 32-column boxes: the first 64 columns in the dS buffer and the rest in the
// staging buffer when D = 128; all of it in the staging buffer when D = 64.
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

template <int DT>
struct Elem;
template <>
struct Elem<kDtBF16> {
  using T = __nv_bfloat16;
  static constexpr int kAB = 1;
  __device__ static uint32_t pack(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static float2 unpack(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u));
  }
};
template <>
struct Elem<kDtF16> {
  using T = __half;
  static constexpr int kAB = 0;
  __device__ static uint32_t pack(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static float2 unpack(uint32_t u) {
    return __half22float2(*reinterpret_cast<__half2*>(&u));
  }
};

__device__ __forceinline__ void record_error(int* header, int where) {
  atomicCAS(&header[kHdrErrorWhere], 0, where);
  atomicExch(&header[kHdrError], 1);
  atomicAdd(&header[kHdrErrorCounts + (where & 15)], 1);  // every failing wait, by code
}

// Zero rows [r0, 128) of a [128 x 64*panels] swizzled tile (full 128-byte rows,
// so the swizzle does not matter). Executed by one warp.
__device__ __forceinline__ void zero_rows(uint8_t* tile, int panels, int r0, int lane) {
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

template <int D, int DT>
__global__ void __launch_bounds__(kThreads, 1)
    k_bwd(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
          const __grid_constant__ CUtensorMap tm_acc, const Plan p) {
  using S = Smem<D>;
  using E = Elem<DT>;
  using T = typename E::T;
  constexpr int kPanels = D / 64;
  constexpr uint32_t kIdS = idesc_f16(128, 128, E::kAB, 0, 0);   // S^T, dP^T
  constexpr uint32_t kIdKV = idesc_f16(128, D, E::kAB, 0, 1);    // dV, dK (A in TMEM)
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
    mbar_init(&bars[kKvTma], 1);
    mbar_init(&bars[kKvFull], 1);
    mbar_init(&bars[kKvEmpty], 1);
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
    mbar_init(&bars[kDkDone], 1);
    mbar_init(&bars[kDqFull], 1);
    mbar_init(&bars[kDqEmpty], 4);
    mbar_init(&bars[kDsFree], 4);  // each drain warp: its dQ boxes in the dS buffer were read
    mbar_init(&bars[kAccFull], 1);
    mbar_init(&bars[kAccEmpty], 4);
    mbar_init(&bars[kItemFull0], 1);
    mbar_init(&bars[kItemFull1], 1);
    mbar_init(&bars[kItemEmpty0], 13);
    mbar_init(&bars[kItemEmpty1], 13);
    mbar_init(&bars[kDrainBar], 1);
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

  uint8_t* sK = smem + S::oK;
  uint8_t* sV = smem + S::oV;
  uint8_t* sQ0 = smem + S::oQ;
  uint8_t* sdO = smem + S::odO;
  uint8_t* sdS = smem + S::odS;
  uint8_t* sStg = smem + S::oStg;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    uint32_t n = 0, itc = 0;
    uint32_t aux_cnt[2] = {0u, 0u}, do_aux_cnt = 0;
    uint32_t last_q_par[2] = {0u, 0u}, last_do_par = 0;
    int pending_q[2] = {0, 0}, pending_q_aux[2] = {0, 0};
    int pending_do = 0, pending_do_aux = 0;
    int pending_kv = 0;
    bool ok = true;
    while (ok) {
      const int slot = itc & 1;
      if (!mbar_wait(&bars[kItemEmpty0 + slot], ((itc >> 1) & 1) ^ 1, abort_flag)) {
        record_error(p.header, kErrWaitItem);
        break;
      }
      if (lane == 0) {
        const int idx = atomicAdd(&p.header[kHdrWorkCounter], 1);
        int4 it = make_int4(-1, 0, 0, -1);
        if (idx < p.header[kHdrNumItems]) it = p.items[idx];
        item_slot[slot] = it;
        mbar_arrive(&bars[kItemFull0 + slot]);
      }
      __syncwarp();
      const int4 raw = item_slot[slot];
      if (raw.x < 0) break;
      const ItemInfo ii = decode_item(p, raw);
      if (ii.e0 >= ii.e1) { ++itc; continue; }
      const int Lq = p.lq[ii.b], Lk = p.lk[ii.b];
      const int t_valid = Lk - ii.jt * 128;
      if (!mbar_wait(&bars[kKvEmpty], (itc & 1) ^ 1, abort_flag)) {
        record_error(p.header, kErrWaitKV);
        break;
      }
      pending_kv = 1;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[kKvTma], 2u * S::kTileBytes);
        const int c1 = p.layout == kLayoutBNSD ? ii.jt * 128 : ii.g;
        const int c2 = p.layout == kLayoutBNSD ? ii.b * p.N2 + ii.g : p.cu_k[ii.b] + ii.jt * 128;
        const uint64_t pol = l2_policy_evict_first();  // K/V: read once per item
        for (int pn = 0; pn < kPanels; ++pn) {
          tma_load_3d_hint(sK + pn * kPanel, &tm_k, &bars[kKvTma], pn * 64, c1, c2, pol);
          tma_load_3d_hint(sV + pn * kPanel, &tm_v, &bars[kKvTma], pn * 64, c1, c2, pol);
        }
      }
      for (int e = ii.e0; e < ii.e1 && ok; ++e) {
        const int32_t ent = p.entries[e];
        const int it = entry_it(ent);
        const int h = ii.g * p.G + entry_hl(ent);
        const int st = n & 1;
        const int q0 = it * 128;
        const bool tail = (Lq - q0) < 128;
        const int c1 = p.layout == kLayoutBNSD ? q0 : h;
        const int c2 = p.layout == kLayoutBNSD ? ii.b * p.N1 + h : p.cu_q[ii.b] + q0;
        // Q (stage st) with its lse / D rows
        if (!mbar_wait(&bars[kQEmpty0 + st], ((n >> 1) & 1) ^ 1, abort_flag)) {
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
          reinterpret_cast<float4*>(sLse + st * 128)[lane] = l4;
          reinterpret_cast<float4*>(sDv + st * 128)[lane] = d4;
        }
        __syncwarp();
        if (tail) {
          if (!mbar_wait(&bars[kQAux0 + st], aux_cnt[st] & 1, abort_flag)) {
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
        // dO (single buffer): free once the previous tile's dV MMA completed
        if (!mbar_wait(&bars[kDoEmpty], (n & 1) ^ 1, abort_flag)) {
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
          if (!mbar_wait(&bars[kDoAux], do_aux_cnt & 1, abort_flag)) {
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
        if (e == ii.e0) {
          // K/V of this item: wait for the copy, clear rows past the key length
          if (!mbar_wait(&bars[kKvTma], itc & 1, abort_flag)) {
            record_error(p.header, kErrWaitKV);
            ok = false;
            break;
          }
          pending_kv = 0;
          if (t_valid < 128) {
            zero_rows(sK, kPanels, t_valid, lane);
            zero_rows(sV, kPanels, t_valid, lane);
            fence_async_smem();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kKvFull]);
        }
        ++n;
      }
      ++itc;
    }
    if (*abort_flag) {
      // let copies still in flight land before the CTA exits
      for (int st = 0; st < 2; ++st) {
        if (pending_q[st]) mbar_wait_drain(&bars[kQFull0 + st], last_q_par[st]);
        if (pending_q_aux[st]) mbar_wait_drain(&bars[kQAux0 + st], aux_cnt[st] & 1);
      }
      if (pending_do) mbar_wait_drain(&bars[kDoFull], last_do_par);
      if (pending_do_aux) mbar_wait_drain(&bars[kDoAux], do_aux_cnt & 1);
      if (pending_kv) mbar_wait_drain(&bars[kKvTma], (itc & 1));
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    uint32_t n = 0, itc = 0;
    const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), adS = smem_u32(sdS);
    int where = 0;
    while (true) {
      const int slot = itc & 1;
      if (!mbar_wait(&bars[kItemFull0 + slot], (itc >> 1) & 1, abort_flag)) { where = kErrWaitItem; break; }
      const int4 raw = item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + slot]);
      if (raw.x < 0) break;
      const ItemInfo ii = decode_item(p, raw);
      if (ii.e0 >= ii.e1) { ++itc; continue; }
      // test of the bounded waits: a barrier no one arrives at runs out, the CTA
      // unwinds and the host reads the error code
      if (p.wait_test && !mbar_wait(&bars[kNeverBar], 0, abort_flag)) { where = kErrWaitTest; break; }
      if (!mbar_wait(&bars[kKvFull], itc & 1, abort_flag)) { where = kErrWaitKV; break; }
      tc_fence_after();
      bool first = true;
      for (int e = ii.e0; e < ii.e1; ++e) {
        const int st = n & 1;
        const uint32_t aQ = smem_u32(sQ0 + st * S::kTileBytes);
        const uint32_t adO = smem_u32(sdO);
        if (!mbar_wait(&bars[kQFull0 + st], (n >> 1) & 1, abort_flag)) { where = kErrWaitQ; break; }
        tc_fence_after();
        if (lane == 0) {  // S^T = K Q^T
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * kPanel + (k & 3) * 32;
            mma_ss(tmem + kColS, sdesc_sw128(aK + off, 16, 1024), sdesc_sw128(aQ + off, 16, 1024),
                   kIdS, k > 0);
          }
          tc_commit(&bars[kSFull]);
        }
        __syncwarp();
        if (!mbar_wait(&bars[kDqEmpty], (n & 1) ^ 1, abort_flag)) { where = kErrWaitDQ; break; }
        if (!mbar_wait(&bars[kDoFull], n & 1, abort_flag)) { where = kErrWaitQ; break; }
        tc_fence_after();
        if (lane == 0) {  // dP^T = V dO^T
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * kPanel + (k & 3) * 32;
            mma_ss(tmem + kColP, sdesc_sw128(aV + off, 16, 1024), sdesc_sw128(adO + off, 16, 1024),
                   kIdS, k > 0);
          }
          tc_commit(&bars[kDpFull]);
        }
        __syncwarp();
        if (!mbar_wait(&bars[kPReady], n & 1, abort_flag)) { where = kErrWaitP; break; }
        // the first dV/dK MMAs of an item overwrite the accumulators: the drain
        // warps must have read the previous item's dK/dV
        if (first && !mbar_wait(&bars[kAccEmpty], (itc & 1) ^ 1, abort_flag)) { where = kErrWaitAcc; break; }
        tc_fence_after();
        if (lane == 0) {  // dV^T += P^T dO  (A = P^T in TMEM, packed)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t acol = kColS + 64 * (k >> 2) + 8 * (k & 3);
            mma_ts(tmem + kColDV, tmem + acol, sdesc_sw128(adO + k * 2048, kPanel, 1024), kIdKV,
                   (first && k == 0) ? 0u : 1u);
          }
          tc_commit(&bars[kDoEmpty]);  // dO may be reloaded once dP and dV completed
        }
        __syncwarp();
        if (!mbar_wait(&bars[kDsReady], n & 1, abort_flag)) { where = kErrWaitDS; break; }
        tc_fence_after();
        if (lane == 0) {  // dK^T += dS^T Q  (A = dS^T in TMEM, packed)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t acol = kColP + 64 * (k >> 2) + 8 * (k & 3);
            mma_ts(tmem + kColDK, tmem + acol, sdesc_sw128(aQ + k * 2048, kPanel, 1024), kIdKV,
                   (first && k == 0) ? 0u : 1u);
          }
          tc_commit(&bars[kDkDone]);
          tc_commit(&bars[kQEmpty0 + st]);
        }
        __syncwarp();
        // dQ reuses the dS^T columns: wait until the dK MMAs have read them
        if (!mbar_wait(&bars[kDkDone], n & 1, abort_flag)) { where = kErrWaitMisc; break; }
        tc_fence_after();
        if (lane == 0) {  // dQ = dS K  (A = dS from smem, MN-major; B = K, MN-major)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            mma_ss(tmem + kColP, sdesc_sw128(adS + k * 2048, kPanel, 1024),
                   sdesc_sw128(aK + k * 2048, kPanel, 1024), kIdQ, k > 0);
          }
          tc_commit(&bars[kDqFull]);
        }
        __syncwarp();
        first = false;
        ++n;
      }
      if (where) break;
      if (lane == 0) {
        tc_commit(&bars[kAccFull]);
        tc_commit(&bars[kKvEmpty]);
      }
      __syncwarp();
      ++itc;
    }
    if (where) record_error(p.header, where);
    if (*abort_flag) {  // wait for MMAs still in flight before TMEM is freed
      if (lane == 0) tc_commit(&bars[kDrainBar]);
      __syncwarp();
      mbar_wait_drain(&bars[kDrainBar], 0);
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
      if (!mbar_wait(&bars[kItemFull0 + slot], (itc >> 1) & 1, abort_flag)) { where = kErrWaitItem; break; }
      const int4 raw = item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + slot]);
      if (raw.x < 0) break;
      const ItemInfo ii = decode_item(p, raw);
      if (ii.e0 >= ii.e1) { ++itc; continue; }
      const int Lq = p.lq[ii.b], Lk = p.lk[ii.b];
      const bool t_ok = (ii.jt * 128 + t) < Lk;
      for (int e = ii.e0; e < ii.e1; ++e) {
        const int32_t ent = p.entries[e];
        const int it = entry_it(ent);
        const int sub = entry_sub(ent);
        const int s_sub = (p.rb == 2) ? wg : 0;
        const int t_sub = (p.cb == 2) ? (t >> 6) : 0;
        const bool row_on = t_ok && ((sub >> (s_sub * 2 + t_sub)) & 1);
        const int s_lim = Lq - it * 128;
        const int st = n & 1;
        if (!mbar_wait(&bars[kQFull0 + st], (n >> 1) & 1, abort_flag)) { where = kErrWaitQ; break; }
        if (!mbar_wait(&bars[kSFull], n & 1, abort_flag)) { where = kErrWaitS; break; }
        tc_fence_after();
        const float* lse2 = sLse + st * 128;
        const float* dv = sDv + st * 128;
        // P^T of this thread's 64 columns, packed to the operand type (the
        // same rounded values feed the dV MMA and dS = P o (dP - D))
        uint32_t Ppk[32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t x[32];
          tmem_ld32(tmem + lane_off + kColS + 64 * wg + 32 * c, x);
          const int s0 = 64 * wg + 32 * c;
          const bool full = row_on && (s_lim >= s0 + 32);
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 l4 = reinterpret_cast<const float4*>(lse2 + s0)[j4];
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
            float pv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int j = 4 * j4 + u;
              pv[u] = ex2_approx(fmaf(__uint_as_float(x[j]), p.scale_log2, -lv[u]));
              if (!full) pv[u] = (row_on && (s0 + j) < s_lim) ? pv[u] : 0.f;
            }
            Ppk[16 * c + 2 * j4] = E::pack(pv[0], pv[1]);
            Ppk[16 * c + 2 * j4 + 1] = E::pack(pv[2], pv[3]);
          }
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = Ppk[16 * c + j];
          tmem_st16(tmem + lane_off + kColS + 64 * wg + 16 * c, pk);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kPReady]);
        if (!mbar_wait(&bars[kDpFull], n & 1, abort_flag)) { where = kErrWaitDP; break; }
        if (!mbar_wait(&bars[kDsFree], (n & 1) ^ 1, abort_flag)) { where = kErrWaitMisc; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t y[32];
          tmem_ld32(tmem + lane_off + kColP + 64 * wg + 32 * c, y);
          const int s0 = 64 * wg + 32 * c;
          uint32_t pk[16];
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 d4 = reinterpret_cast<const float4*>(dv + s0)[j4];
            const float dd[4] = {d4.x, d4.y, d4.z, d4.w};
            float ds[4];
            const float2 p01 = E::unpack(Ppk[16 * c + 2 * j4]);
            const float2 p23 = E::unpack(Ppk[16 * c + 2 * j4 + 1]);
            ds[0] = p01.x * (__uint_as_float(y[4 * j4 + 0]) - dd[0]);
            ds[1] = p01.y * (__uint_as_float(y[4 * j4 + 1]) - dd[1]);
            ds[2] = p23.x * (__uint_as_float(y[4 * j4 + 2]) - dd[2]);
            ds[3] = p23.y * (__uint_as_float(y[4 * j4 + 3]) - dd[3]);
            pk[2 * j4] = E::pack(ds[0], ds[1]);
            pk[2 * j4 + 1] = E::pack(ds[2], ds[3]);
          }
          tmem_st16(tmem + lane_off + kColP + 64 * wg + 16 * c, pk);
          // dS (M = query s, K = key t) for the dQ MMA: panel wg, row t,
          // 16-byte chunk cc holds s = 64 wg + 8 cc .. +7, swizzled by t & 7.
          uint8_t* rowp = sdS + wg * kPanel + t * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int cc = 4 * c + q;
            *reinterpret_cast<uint4*>(rowp + ((cc ^ (t & 7)) << 4)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
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
    // -------------------------------------------------------------- drain
    const int qd = warp & 3;
    const int r = qd * 32 + lane;  // TMEM lane: query row (dQ) / key row (dK, dV)
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    uint32_t n = 0, itc = 0;
    int where = 0;
    while (true) {
      const int slot = itc & 1;
      if (!mbar_wait(&bars[kItemFull0 + slot], (itc >> 1) & 1, abort_flag)) { where = kErrWaitItem; break; }
      const int4 raw = item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + slot]);
      if (raw.x < 0) break;
      const ItemInfo ii = decode_item(p, raw);
      if (ii.e0 >= ii.e1) { ++itc; continue; }
      const int Lq = p.lq[ii.b], Lk = p.lk[ii.b];
      for (int e = ii.e0; e < ii.e1; ++e) {
        const int32_t ent = p.entries[e];
        const int it = entry_it(ent);
        const int h = ii.g * p.G + entry_hl(ent);
        if (!mbar_wait(&bars[kDqFull], n & 1, abort_flag)) { where = kErrWaitDQ; break; }
        tc_fence_after();
        // dQ tile -> fp32 accumulator with TMA reduce-adds. Each warp copies its
        // 32 rows from TMEM into 32x32 fp32 boxes (128-byte swizzled): columns
        // [0, 64) into the dS buffer and [64, 128) into the staging buffer
        // when D = 128 (D = 64: staging buffer only), releases TMEM for the
        // next dP, and issues the reduce-adds as two bulk groups. The dS half
        // must be read before the softmax warps write the next dS (ds_free);
        // the staging half is waited for before this warp stages again. Rows
        // past the query length carry exact zeros (dS = 0 there) and land in
        // the padded part of the accumulator.
        const int grow = h * p.Rq + p.qrow[ii.b] + it * 128 + qd * 32;
        uint8_t* boxes_ds = sdS + qd * 8192;
        uint8_t* boxes_stg = sStg + qd * 8192;
        if (lane == 0) bulk_wait_read_all();  // previous tile's staging boxes were read
        __syncwarp();
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf) {
          uint8_t* boxes = (D == 128 && hf == 0) ? boxes_ds : boxes_stg;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t x[32];
            tmem_ld32(tmem + lane_off + kColP + 64 * hf + 32 * c, x);
            uint8_t* rowp = boxes + c * 4096 + lane * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) =
                  make_uint4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
          }
        }
        tc_fence_before();
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars[kDqEmpty]);  // TMEM columns free for the next dP
          const uint64_t pol = l2_policy_evict_last();  // keep dQ accumulator rows in L2
          if (D == 128) {
            tma_reduce_add_2d_hint(&tm_acc, boxes_ds, 0, grow, pol);
            tma_reduce_add_2d_hint(&tm_acc, boxes_ds + 4096, 32, grow, pol);
            bulk_commit_group();
            tma_reduce_add_2d_hint(&tm_acc, boxes_stg, 64, grow, pol);
            tma_reduce_add_2d_hint(&tm_acc, boxes_stg + 4096, 96, grow, pol);
            bulk_commit_group();
            bulk_wait_read_1();                 // the dS-buffer group has been read
          } else {
            tma_reduce_add_2d_hint(&tm_acc, boxes_stg, 0, grow, pol);
            tma_reduce_add_2d_hint(&tm_acc, boxes_stg + 4096, 32, grow, pol);
            bulk_commit_group();
          }
          mbar_arrive(&bars[kDsFree]);
        }
        __syncwarp();
        ++n;
      }
      if (where) break;
      // dK / dV of the key tile
      if (!mbar_wait(&bars[kAccFull], itc & 1, abort_flag)) { where = kErrWaitAcc; break; }
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
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? kColDK : kColDV;
        const float mul = which == 0 ? p.scale : 1.f;
        T* out = static_cast<T*>(which == 0 ? p.dk : p.dv) + (which == 0 ? ok_off : ov_off);
        const int64_t sd = which == 0 ? sdk : sdv;
#pragma unroll
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
      ++itc;
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

template <int D, int DT>
cudaError_t launch_t(const Plan& p, const BwdMaps& m, cudaStream_t st) {
  const size_t smem = Smem<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(k_bwd<D, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  int grid = p.num_sms;
  if (p.max_items < grid) grid = p.max_items;
  if (grid < 1) grid = 1;
  k_bwd<D, DT><<<grid, kThreads, smem, st>>>(m.q, m.k, m.v, m.dout, m.dqacc, p);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_smem_bytes(int D) { return D == 128 ? Smem<128>::kBytes : Smem<64>::kBytes; }

cudaError_t launch_bwd(const Plan& p, const BwdMaps& m, cudaStream_t st) {
  if (p.dtype == kDtBF16)
    return p.D == 128 ? launch_t<128, kDtBF16>(p, m, st) : launch_t<64, kDtBF16>(p, m, st);
  return p.D == 128 ? launch_t<128, kDtF16>(p, m, st) : launch_t<64, kDtF16>(p, m, st);
}

}  // namespace bsa
