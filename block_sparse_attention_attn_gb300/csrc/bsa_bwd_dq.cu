// bsa_bwd_dq.cu - deterministic dQ pass of the block-sparse attention backward
// on the sm_103a tensor cores. For every query tile it walks the selected key
// tiles in ascending order and accumulates
//     dQ = scale * sum_j dS_j K_j,   dS_j = P_j o (dP_j - D),
//     P_j = exp(scale * Q K_j^T - lse),   dP_j = dO V_j^T
// (backward formulas of the aclnnBlockSparseAttentionGrad page, section
// 计算公式) in TMEM, so the result does not depend on the order in which
// other CTAs finish: no fp32 reduce-adds, the same bits on every run. The
// key-tile-stationary kernel then computes dK and dV only.
//
// One persistent CTA per SM, 384 threads:
//   warp 8      producer: Q and dO of the query tile, then K and V tiles of
//               the selected key tiles (found by scanning the mask row)
//               through TMA rings of 3 (K: read by S and the later dQ) and
//               2 (V: read by dP only) stages;
//   warp 9      MMA issuer of S(m) = Q K^T (into one of two S buffers) and
//               dP(m) = dO V^T (once the softmax warps have read dP(m-1)),
//               and TMEM owner;
//   warp 10     MMA issuer of dQ += dS(m) K(m) (dS read from TMEM) as soon as
//               the softmax warps have written dS(m): the tensor cores compute
//               tile m+1 while the softmax warps work on tile m, and neither
//               issuer waits behind the other's issue (an issuing thread
//               blocks while the tensor pipe's queue is full);
//   warps 0-7   two warpgroups, TMEM lane s = query row s, warpgroup wg owns
//               keys [64 wg, 64 wg + 64): P and dS (lse and D are per-thread
//               values here), then the dQ epilogue (columns split by wg).
// TMEM columns: [0,128) and [128,256) S, with dS packed in place (keys 0-63
// at the buffer's columns [0,32), keys 64-127 at [96,128), so neither
// warpgroup overwrites S values the other still reads); [256,384) dP;
// [384,384+D) dQ.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bsa_common.h"
#include "bsa_launch.h"
#include "bsa_device.cuh"
#include "sm103_ptx.cuh"

namespace bsa {
namespace {

constexpr int kThreads = 384;
constexpr int kSoftmaxWarps = 8;
constexpr int kProdWarp = 8;
constexpr int kMmaWarp = 9;   // S, dP; TMEM owner
constexpr int kDqWarp = 10;   // dQ; warp 11 only lends its registers
// Registers per thread after the hand-over (launch: 384 x 168): the control
// warpgroup (warps 8-11) keeps 64, the two softmax warpgroups get 208 each.
// Each budget has its own copy of the out-of-line wait loop (wait tags).
constexpr int kRegsLaunch = 168, kRegsCtl = 64, kRegsSoftmax = 208;
constexpr int kTagCtl = 1, kTagSoftmax = 2;
constexpr int kPanel = 128 * 128;
constexpr uint32_t kColS0 = 0, kColP = 256, kColQ = 384;
constexpr int kKStages = 3, kVStages = 2;

// TMEM column of the packed dS of keys [16 kk, 16 kk + 16) inside an S buffer.
__host__ __device__ constexpr uint32_t ds_col(int kk) { return (kk >> 2) * 96 + (kk & 3) * 8; }

enum Bar {
  kQFull = 0, kQAux, kQEmpty,
  kKFull0, kKFull1, kKFull2, kKEmpty0, kKEmpty1, kKEmpty2, kKAux0, kKAux1, kKAux2,
  kVFull0, kVFull1, kVEmpty0, kVEmpty1, kVAux0, kVAux1,
  kSFull0, kSFull1, kSFree0, kSFree1, kDpFull, kDpFree, kDsReady, kDqFull, kDqEmpty,
  kItemFull0, kItemFull1, kItemEmpty0, kItemEmpty1,
  kDrain, kDrain2,
  kNumBars
};

template <int D>
struct Smem {
  static constexpr int kTileBytes = (D / 64) * kPanel;
  static constexpr int oQ = 0;
  static constexpr int odO = oQ + kTileBytes;
  static constexpr int oK = odO + kTileBytes;             // [kKStages]
  static constexpr int oV = oK + kKStages * kTileBytes;   // [kVStages]
  static constexpr int oBar = oV + kVStages * kTileBytes;
  static constexpr int oMisc = (oBar + kNumBars * 8 + 63) / 64 * 64;
  static_assert(oMisc % 16 == 0, "misc area must be 16-byte aligned");
  static constexpr int kBytes = oMisc + 128;
};

__device__ __forceinline__ void zero_rows(uint8_t* tile, int panels, int r0, int lane) {
  const int n16 = (128 - r0) * 8;
  for (int pnl = 0; pnl < panels; ++pnl) {
    uint4* base = reinterpret_cast<uint4*>(tile + pnl * kPanel + r0 * 128);
    for (int i = lane; i < n16; i += 32) base[i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Packed fp32 pairs (two lanes of one 64-bit register): one instruction for
// two columns of the P and dS loops.
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

struct QItem {
  int b, h, it;
};

__device__ __forceinline__ QItem decode(const Plan& p, int idx) {
  QItem r;
  r.it = idx % p.Mq_t;
  const int bh = idx / p.Mq_t;
  r.h = bh % p.N1;
  r.b = bh / p.N1;
  return r;
}

// Sub-block bits of key tile jt for query tile it of (b, h); 0 when the tile
// has no selected block inside the valid range that meets the sliding window.
__device__ __forceinline__ int q_tile_bits(const Plan& p, int b, int h, int it, int jt, int Lq, int Lk) {
  int bits = 0;
  for (int ri = 0; ri < p.rb; ++ri) {
    const int i = it * p.rb + ri;
    if (i * p.bx >= Lq) break;
    for (int cj = 0; cj < p.cb; ++cj) {
      const int j = jt * p.cb + cj;
      if (j * p.by >= Lk) break;
      bool on = true;
      if (p.has_mask)
        on = (i < p.Mq && j < p.Mk) &&
             p.mask[(int64_t)b * p.mask_sb + (int64_t)h * p.mask_sh + (int64_t)i * p.mask_si + j] != 0;
      if (on && p.win)
        on = win_meets((int64_t)i * p.bx, min((int64_t)(i + 1) * p.bx, (int64_t)Lq),
                       (int64_t)j * p.by, min((int64_t)(j + 1) * p.by, (int64_t)Lk), p.win_pre,
                       p.win_next);
      if (on && p.am) on = am_block_meets(p.am_sub, p.am_sk, i, j, p.bx, p.by);
      if (on) bits |= 1 << (ri * 2 + cj);
    }
  }
  return bits;
}

template <int D, int DT>
__global__ void __launch_bounds__(kThreads, 1)
    k_bwd_dq(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
             const Plan p) {
  using S = Smem<D>;
  using E = Elem<DT>;
  using T = typename E::T;
  constexpr int kPanels = D / 64;
  constexpr uint32_t kIdS = idesc_f16(128, 128, E::kAB, 0, 0);  // S = Q K^T, dP = dO V^T
  constexpr uint32_t kIdQ = idesc_f16(128, D, E::kAB, 0, 1);     // dQ += dS K (A in TMEM)

  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::oBar);
  int* misc = reinterpret_cast<int*>(smem + S::oMisc);
  volatile int* abort_flag = misc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 1);
  int* item_slot = misc + 2;  // [2]
  int* meta = misc + 4;       // [kKStages] per K stage: jt | bits << 24, -1 = end of item
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(p.header, kErrSmemAlign);
    return;
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(&bars[kQFull], 1);
    mbar_init(&bars[kQAux], 1);
    mbar_init(&bars[kQEmpty], 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&bars[kKFull0 + i], 1);
      mbar_init(&bars[kKEmpty0 + i], 2 + kSoftmaxWarps);  // both MMA warps (commit or arrive) + softmax warps
      mbar_init(&bars[kKAux0 + i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&bars[kVFull0 + i], 1);
      mbar_init(&bars[kVEmpty0 + i], 1);  // dP MMA commit
      mbar_init(&bars[kVAux0 + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kItemFull0 + i], 1);
      mbar_init(&bars[kItemEmpty0 + i], 2 + kSoftmaxWarps);
      mbar_init(&bars[kSFull0 + i], 1);   // S MMA commit
      mbar_init(&bars[kSFree0 + i], 1);   // dQ MMA commit: the buffer's dS was read
    }
    mbar_init(&bars[kDpFull], 1);
    mbar_init(&bars[kDpFree], kSoftmaxWarps);   // dP read out of TMEM
    mbar_init(&bars[kDsReady], kSoftmaxWarps);
    mbar_init(&bars[kDqFull], 1);
    mbar_init(&bars[kDqEmpty], kSoftmaxWarps);
    mbar_init(&bars[kDrain], 1);
    mbar_init(&bars[kDrain2], 1);
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == kProdWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  uint8_t* sQ = smem + S::oQ;
  uint8_t* sdO = smem + S::odO;
  uint8_t* sK0 = smem + S::oK;
  uint8_t* sV0 = smem + S::oV;
  const int n_items = p.B * p.N1 * p.Mq_t;

  if (warp >= kProdWarp) {
  regs_release<kRegsCtl>();  // all four warps of the control warpgroup
  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    uint32_t nk = 0, nv = 0, itc = 0, qaux = 0;  // K stages (end markers included), V stages
    uint32_t kaux[kKStages] = {0u, 0u, 0u}, vaux[kVStages] = {0u, 0u};
    bool ok = true;
    int pend_q = 0, pend_qaux = 0;
    int pend_k[kKStages] = {0, 0, 0}, pend_kaux[kKStages] = {0, 0, 0};
    int pend_v[kVStages] = {0, 0}, pend_vaux[kVStages] = {0, 0};
    uint32_t par_k[kKStages] = {0u, 0u, 0u}, par_v[kVStages] = {0u, 0u};
    while (ok) {
      const int slot = itc & 1;
      if (!mbar_wait<kTagCtl>(&bars[kItemEmpty0 + slot], ((itc >> 1) & 1) ^ 1, abort_flag)) {
        record_error(p.header, kErrWaitItem);
        break;
      }
      if (lane == 0) {
        const int idx = atomicAdd(&p.header[kHdrDqCounter], 1);
        item_slot[slot] = idx < n_items ? idx : -1;
        mbar_arrive(&bars[kItemFull0 + slot]);
      }
      __syncwarp();
      const int idx = item_slot[slot];
      if (idx < 0) break;
      const QItem qi = decode(p, idx);
      const int Lq = p.lq[qi.b], Lk = p.lk[qi.b];
      const int q0 = qi.it * 128;
      const bool has_rows = q0 < Lq;
      // Q and dO of the query tile (rows past the query length cleared)
      if (!mbar_wait<kTagCtl>(&bars[kQEmpty], (itc & 1) ^ 1, abort_flag)) {
        record_error(p.header, kErrWaitQ);
        break;
      }
      const bool qtail = (Lq - q0) < 128;
      if (lane == 0) {
        uint64_t* tb = qtail ? &bars[kQAux] : &bars[kQFull];
        mbar_arrive_expect_tx(tb, 2 * S::kTileBytes);
        const int c1 = p.layout == kLayoutBNSD ? q0 : qi.h;
        const int c2 = p.layout == kLayoutBNSD ? qi.b * p.N1 + qi.h : p.cu_q[qi.b] + q0;
        for (int pn = 0; pn < kPanels; ++pn) {
          tma_load_3d(sQ + pn * kPanel, &tm_q, tb, pn * 64, c1, c2);
          tma_load_3d(sdO + pn * kPanel, &tm_do, tb, pn * 64, c1, c2);
        }
      }
      pend_q = qtail ? 0 : 1;
      pend_qaux = qtail ? 1 : 0;
      if (qtail) {
        if (!mbar_wait<kTagCtl>(&bars[kQAux], qaux & 1, abort_flag)) {
          record_error(p.header, kErrWaitQ);
          break;
        }
        qaux++;
        pend_qaux = 0;
        const int r0 = Lq - q0 > 0 ? Lq - q0 : 0;
        zero_rows(sQ, kPanels, r0, lane);
        zero_rows(sdO, kPanels, r0, lane);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kQFull]);
      }
      const int ncolt = has_rows ? (Lk + 127) / 128 : 0;
      const int g = qi.h / p.G;
      for (int jt0 = 0; jt0 < ncolt && ok; jt0 += 32) {
        const int jt = jt0 + lane;
        const int bits = jt < ncolt ? q_tile_bits(p, qi.b, qi.h, qi.it, jt, Lq, Lk) : 0;
        unsigned ball = __ballot_sync(0xffffffffu, bits != 0);
        while (ball && ok) {
          const int src = __ffs(ball) - 1;
          ball &= ball - 1;
          const int jsel = jt0 + src;
          const int bsel = __shfl_sync(0xffffffffu, bits, src);
          const int kst = nk % kKStages, vst = nv % kVStages;
          if (!mbar_wait<kTagCtl>(&bars[kKEmpty0 + kst], ((nk / kKStages) & 1) ^ 1, abort_flag) ||
              !mbar_wait<kTagCtl>(&bars[kVEmpty0 + vst], ((nv / kVStages) & 1) ^ 1, abort_flag)) {
            record_error(p.header, kErrWaitKV);
            ok = false;
            break;
          }
          const bool tail = (Lk - jsel * 128) < 128;
          uint8_t* sK = sK0 + kst * S::kTileBytes;
          uint8_t* sV = sV0 + vst * S::kTileBytes;
          if (lane == 0) {
            meta[kst] = jsel | (bsel << 24);
            uint64_t* tk = tail ? &bars[kKAux0 + kst] : &bars[kKFull0 + kst];
            uint64_t* tv = tail ? &bars[kVAux0 + vst] : &bars[kVFull0 + vst];
            mbar_arrive_expect_tx(tk, S::kTileBytes);
            mbar_arrive_expect_tx(tv, S::kTileBytes);
            const int c1 = p.layout == kLayoutBNSD ? jsel * 128 : g;
            const int c2 = p.layout == kLayoutBNSD ? qi.b * p.N2 + g : p.cu_k[qi.b] + jsel * 128;
            for (int pn = 0; pn < kPanels; ++pn) {
              tma_load_3d(sK + pn * kPanel, &tm_k, tk, pn * 64, c1, c2);
              tma_load_3d(sV + pn * kPanel, &tm_v, tv, pn * 64, c1, c2);
            }
          }
          pend_k[kst] = tail ? 0 : 1;
          par_k[kst] = (nk / kKStages) & 1;
          pend_v[vst] = tail ? 0 : 1;
          par_v[vst] = (nv / kVStages) & 1;
          if (tail) {  // K and V rows past the key length must be finite zeros
            pend_kaux[kst] = 1;
            pend_vaux[vst] = 1;
            if (!mbar_wait<kTagCtl>(&bars[kKAux0 + kst], kaux[kst] & 1, abort_flag) ||
                !mbar_wait<kTagCtl>(&bars[kVAux0 + vst], vaux[vst] & 1, abort_flag)) {
              record_error(p.header, kErrWaitKV);
              ok = false;
              break;
            }
            kaux[kst]++;
            vaux[vst]++;
            pend_kaux[kst] = 0;
            pend_vaux[vst] = 0;
            zero_rows(sK, kPanels, Lk - jsel * 128, lane);
            zero_rows(sV, kPanels, Lk - jsel * 128, lane);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(&bars[kKFull0 + kst]);
              mbar_arrive(&bars[kVFull0 + vst]);
            }
          }
          ++nk;
          ++nv;
        }
      }
      if (!ok) break;
      // end-of-item marker (a K stage without a copy)
      const int kst = nk % kKStages;
      if (!mbar_wait<kTagCtl>(&bars[kKEmpty0 + kst], ((nk / kKStages) & 1) ^ 1, abort_flag)) {
        record_error(p.header, kErrWaitKV);
        break;
      }
      if (lane == 0) {
        meta[kst] = -1;
        mbar_arrive(&bars[kKFull0 + kst]);
      }
      __syncwarp();
      ++nk;
      ++itc;
    }
    if (*abort_flag) {  // let copies still in flight land before the CTA exits
      if (pend_q) mbar_wait_drain(&bars[kQFull], itc & 1);
      if (pend_qaux) mbar_wait_drain(&bars[kQAux], qaux & 1);
      for (int st = 0; st < kKStages; ++st) {
        if (pend_k[st]) mbar_wait_drain(&bars[kKFull0 + st], par_k[st]);
        if (pend_kaux[st]) mbar_wait_drain(&bars[kKAux0 + st], kaux[st] & 1);
      }
      for (int st = 0; st < kVStages; ++st) {
        if (pend_v[st]) mbar_wait_drain(&bars[kVFull0 + st], par_v[st]);
        if (pend_vaux[st]) mbar_wait_drain(&bars[kVAux0 + st], vaux[st] & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------- MMA issuer: S and dP
    uint32_t nk = 0, nv = 0, itc = 0;  // K stages (end markers included), V stages
    uint32_t m = 0;                    // m: computed key tiles (S buffer m & 1)
    int where = 0;
    const uint32_t aQ = smem_u32(sQ), adO = smem_u32(sdO);
    while (true) {
      const int slot = itc & 1;
      if (!mbar_wait<kTagCtl>(&bars[kItemFull0 + slot], (itc >> 1) & 1, abort_flag)) { where = kErrWaitItem; break; }
      const int idx = item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + slot]);
      if (idx < 0) break;
      if (!mbar_wait<kTagCtl>(&bars[kQFull], itc & 1, abort_flag)) { where = kErrWaitQ; break; }
      while (true) {
        const int st = nk % kKStages;
        if (!mbar_wait<kTagCtl>(&bars[kKFull0 + st], (nk / kKStages) & 1, abort_flag)) { where = kErrWaitKV; break; }
        const int mt = meta[st];
        __syncwarp();
        if (mt < 0) {
          if (lane == 0) {
            mbar_arrive(&bars[kKEmpty0 + st]);
            tc_commit(&bars[kQEmpty]);  // Q and dO: their last readers are issued
          }
          __syncwarp();
          ++nk;
          break;
        }
        const uint32_t sb = kColS0 + 128 * (m & 1);
        // the S buffer is free once the dQ MMA of tile m-2 has read its dS
        if (!mbar_wait<kTagCtl>(&bars[kSFree0 + (m & 1)], ((m >> 1) & 1) ^ 1, abort_flag)) { where = kErrWaitMisc; break; }
        tc_fence_after();
        const uint32_t aK = smem_u32(sK0 + st * S::kTileBytes);
        if (lane == 0) {
          const uint64_t dQk = sdesc_sw128(aQ, 16, 1024), dKk = sdesc_sw128(aK, 16, 1024);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint64_t off = (uint64_t)(((k >> 2) * kPanel + (k & 3) * 32) >> 4);
            mma_ss(tmem + sb, dQk + off, dKk + off, kIdS, k > 0);
          }
          tc_commit(&bars[kSFull0 + (m & 1)]);
          tc_commit(&bars[kKEmpty0 + st]);  // this warp's read of K (S)
        }
        __syncwarp();
        // dP has one buffer: the softmax warps must have read dP(m-1)
        const int vst = nv % kVStages;
        if (!mbar_wait<kTagCtl>(&bars[kDpFree], (m & 1) ^ 1, abort_flag)) { where = kErrWaitDP; break; }
        if (!mbar_wait<kTagCtl>(&bars[kVFull0 + vst], (nv / kVStages) & 1, abort_flag)) { where = kErrWaitKV; break; }
        tc_fence_after();
        if (lane == 0) {
          const uint64_t dOk = sdesc_sw128(adO, 16, 1024);
          const uint64_t dVk = sdesc_sw128(smem_u32(sV0 + vst * S::kTileBytes), 16, 1024);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint64_t off = (uint64_t)(((k >> 2) * kPanel + (k & 3) * 32) >> 4);
            mma_ss(tmem + kColP, dOk + off, dVk + off, kIdS, k > 0);
          }
          tc_commit(&bars[kDpFull]);
          tc_commit(&bars[kVEmpty0 + vst]);  // V is read by dP only
        }
        __syncwarp();
        ++nv;
        ++nk;
        ++m;
      }
      if (where) break;
      ++itc;
    }
    if (where) record_error(p.header, where);
    if (*abort_flag) {
      if (lane == 0) tc_commit(&bars[kDrain]);
      __syncwarp();
      mbar_wait_drain(&bars[kDrain], 0);
    }
  } else if (warp == kDqWarp) {
    // ----------------------------------------------------- MMA issuer: dQ
    uint32_t nk = 0, itc = 0, m = 0;  // as in the S / dP issuer
    int where = 0;
    while (true) {
      const int slot = itc & 1;
      if (!mbar_wait<kTagCtl>(&bars[kItemFull0 + slot], (itc >> 1) & 1, abort_flag)) { where = kErrWaitItem; break; }
      const int idx = item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + slot]);
      if (idx < 0) break;
      int j = 0;
      while (true) {
        const int st = nk % kKStages;
        if (!mbar_wait<kTagCtl>(&bars[kKFull0 + st], (nk / kKStages) & 1, abort_flag)) { where = kErrWaitKV; break; }
        const int mt = meta[st];
        __syncwarp();
        if (mt < 0) {
          if (lane == 0) mbar_arrive(&bars[kKEmpty0 + st]);
          ++nk;
          break;
        }
        if (!mbar_wait<kTagCtl>(&bars[kDsReady], m & 1, abort_flag)) { where = kErrWaitDS; break; }
        // the first dQ MMA of an item overwrites the accumulator: the
        // previous item's epilogue must have read it
        if (j == 0 && !mbar_wait<kTagCtl>(&bars[kDqEmpty], (itc & 1) ^ 1, abort_flag)) { where = kErrWaitAcc; break; }
        tc_fence_after();
        if (lane == 0) {  // dQ += dS(m) K: A = dS in S buffer m & 1 (TMEM), B = K (MN-major)
          const uint64_t dKmn = sdesc_sw128(smem_u32(sK0 + st * S::kTileBytes), kPanel, 1024);
          const uint32_t sb = kColS0 + 128 * (m & 1);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts(tmem + kColQ, tmem + sb + ds_col(k), dKmn + (uint64_t)((k * 2048) >> 4), kIdQ,
                   (j == 0 && k == 0) ? 0u : 1u);
          tc_commit(&bars[kSFree0 + (m & 1)]);
          tc_commit(&bars[kKEmpty0 + st]);  // K read for the last time
        }
        __syncwarp();
        ++j;
        ++nk;
        ++m;
      }
      if (where) break;
      if (j == 0 && !mbar_wait<kTagCtl>(&bars[kDqEmpty], (itc & 1) ^ 1, abort_flag)) {  // once per item
        where = kErrWaitAcc;
        break;
      }
      if (lane == 0) tc_commit(&bars[kDqFull]);
      __syncwarp();
      ++itc;
    }
    if (where) record_error(p.header, where);
    if (*abort_flag) {
      if (lane == 0) tc_commit(&bars[kDrain2]);
      __syncwarp();
      mbar_wait_drain(&bars[kDrain2], 0);
    }
  }
  } else {
    regs_claim<kRegsSoftmax>();
    // ----------------------------------------------------- P, dS, epilogue
    const int qd = warp & 3, wg = warp >> 2;
    const int s = qd * 32 + lane;  // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    uint32_t n = 0, itc = 0, m = 0;
    int where = 0;
    while (true) {
      const int slot = itc & 1;
      if (!mbar_wait<kTagSoftmax>(&bars[kItemFull0 + slot], (itc >> 1) & 1, abort_flag)) { where = kErrWaitItem; break; }
      const int idx = item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + slot]);
      if (idx < 0) break;
      const QItem qi = decode(p, idx);
      const int Lq = p.lq[qi.b], Lk = p.lk[qi.b];
      const int srow = qi.it * 128 + s;
      const bool s_ok = srow < Lq;
      // lse2 = lse * log2(e) (+inf past the query length) and D of this row
      const int64_t prow = (int64_t)qi.h * p.Rq + p.qrow[qi.b] + srow;
      const float lse2 = s_ok ? p.lse2[prow] : 0.f;
      const float dsum = s_ok ? p.dvec[prow] : 0.f;
      const int s_sub = p.rb == 2 ? (s >> 6) : 0;
      const int t_sub = p.cb == 2 ? wg : 0;  // this warpgroup's keys lie in one key block
      int j = 0;
      while (true) {
        const int st = n % kKStages;
        if (!mbar_wait<kTagSoftmax>(&bars[kKFull0 + st], (n / kKStages) & 1, abort_flag)) { where = kErrWaitKV; break; }
        const int mt = meta[st];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kKEmpty0 + st]);
        if (mt < 0) {
          ++n;
          break;
        }
        const int jt = mt & 0xFFFFFF, bits = mt >> 24;
        // live key columns [t_lo, t_hi) of the tile (key length and window),
        // restricted to this warpgroup's 64; amw: token mask bits (set = masked)
        int t_lo = 0, t_hi = Lk - jt * 128;
        if (p.win) {
          const int2 w = win_span(srow, (int64_t)jt * 128, -p.win_pre, p.win_next);
          t_lo = w.x;
          t_hi = min(t_hi, w.y);
        }
        uint2 amw = make_uint2(0u, 0u);
        if (p.am)
          amw = *reinterpret_cast<const uint2*>(p.am_row + (int64_t)srow * p.am_wk + 4 * jt + 2 * wg);
        const bool row_on = s_ok && ((bits >> (s_sub * 2 + t_sub)) & 1);
        const uint32_t live0 = row_on ? bit_range(t_lo - 64 * wg, t_hi - 64 * wg) & ~amw.x : 0u;
        const uint32_t live1 = row_on ? bit_range(t_lo - 64 * wg - 32, t_hi - 64 * wg - 32) & ~amw.y : 0u;
        const uint32_t sb = kColS0 + 128 * (m & 1);
        if (!mbar_wait<kTagSoftmax>(&bars[kSFull0 + (m & 1)], (m >> 1) & 1, abort_flag)) { where = kErrWaitS; break; }
        tc_fence_after();
        // P of this warpgroup's 64 keys, rounded to the operand type as in the
        // dV/dK kernel, kept packed in registers
        uint32_t Ppk[32];
        {
          uint32_t x[64];  // both 32-column chunks in one TMEM load
          tmem_ld64(tmem + lane_off + sb + 64 * wg, x);
          if ((live0 & live1) == 0xFFFFFFFFu) {  // every key takes part: no per-key tests
            const uint64_t c2 = f2(__float_as_uint(p.scale_log2), __float_as_uint(p.scale_log2));
            const uint64_t nl2 = f2(__float_as_uint(-lse2), __float_as_uint(-lse2));
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              float t0, t1;
              f2split(fma2(f2(x[2 * k], x[2 * k + 1]), c2, nl2), t0, t1);
              Ppk[k] = E::pack(ex2_approx(t0), ex2_approx(t1));
            }
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const uint32_t live = k < 16 ? live0 : live1;
              float pv[2];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const bool on = (live >> ((2 * k + u) & 31)) & 1u;
                pv[u] = on ? ex2_approx(fmaf(__uint_as_float(x[2 * k + u]), p.scale_log2, -lse2)) : 0.f;
              }
              Ppk[k] = E::pack(pv[0], pv[1]);
            }
          }
        }
        if (!mbar_wait<kTagSoftmax>(&bars[kDpFull], m & 1, abort_flag)) { where = kErrWaitDP; break; }
        tc_fence_after();
        uint32_t y[64];
        tmem_ld64(tmem + lane_off + kColP + 64 * wg, y);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kDpFree]);  // the MMA may write dP(m+1)
        // dS = P o (dP - D), packed in place over this warpgroup's S columns
        {
          uint32_t pk[32];
          const uint64_t d2 = f2(__float_as_uint(dsum), __float_as_uint(dsum));
#pragma unroll
          for (int k = 0; k < 32; ++k) {  // two columns per packed subtract and multiply
            const float2 pp = E::unpack(Ppk[k]);
            float a0, a1;
            f2split(mul2(sub2(f2(y[2 * k], y[2 * k + 1]), d2), f2(__float_as_uint(pp.x), __float_as_uint(pp.y))),
                    a0, a1);
            pk[k] = E::pack(a0, a1);
          }
          tmem_st32(tmem + lane_off + sb + 96 * wg, pk);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kDsReady]);
        ++j;
        ++n;
        ++m;
      }
      if (where) break;
      // epilogue: dQ = scale * accumulator (zeros when no key tile was
      // selected); warpgroup wg writes the columns [wg D/2, wg D/2 + D/2)
      if (!mbar_wait<kTagSoftmax>(&bars[kDqFull], itc & 1, abort_flag)) { where = kErrWaitAcc; break; }
      tc_fence_after();
      const bool write_row = p.layout == kLayoutBNSD ? (srow < p.Sq) : s_ok;
      int64_t ooff, sd;
      if (p.layout == kLayoutBNSD) {
        ooff = qi.b * p.dq_st[0] + qi.h * p.dq_st[1] + (int64_t)srow * p.dq_st[2];
        sd = p.dq_st[3];
      } else {
        ooff = ((int64_t)p.cu_q[qi.b] + srow) * p.dq_st[0] + qi.h * p.dq_st[1];
        sd = p.dq_st[2];
      }
      T* out = static_cast<T*>(p.dq) + ooff;
      const float mul = (s_ok && j > 0) ? p.scale : 0.f;
#pragma unroll 1
      for (int c = wg * (D / 64); c < (wg + 1) * (D / 64); ++c) {
        uint32_t o[32];
        if (j > 0) {
          tmem_ld32(tmem + lane_off + kColQ + 32 * c, o);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = 0u;
        }
        if (write_row) {
          if (p.dq_vec) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 u;
              u.x = E::pack(__uint_as_float(o[8 * q]) * mul, __uint_as_float(o[8 * q + 1]) * mul);
              u.y = E::pack(__uint_as_float(o[8 * q + 2]) * mul, __uint_as_float(o[8 * q + 3]) * mul);
              u.z = E::pack(__uint_as_float(o[8 * q + 4]) * mul, __uint_as_float(o[8 * q + 5]) * mul);
              u.w = E::pack(__uint_as_float(o[8 * q + 6]) * mul, __uint_as_float(o[8 * q + 7]) * mul);
              *reinterpret_cast<uint4*>(out + 32 * c + 8 * q) = u;
            }
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const uint32_t pk = E::pack(__uint_as_float(o[k]) * mul, 0.f);
              out[(32 * c + k) * sd] = *reinterpret_cast<const T*>(&pk);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kDqEmpty]);
      ++itc;
    }
    if (where) record_error(p.header, where);
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
  // The register hand-over only balances when every thread starts with
  // kRegsLaunch registers.
  static const int regs = [] {
    cudaFuncAttributes fa{};
    return cudaFuncGetAttributes(&fa, k_bwd_dq<D, DT>) == cudaSuccess ? fa.numRegs : -1;
  }();
  static_assert(2 * kRegsSoftmax + kRegsCtl <= 3 * kRegsLaunch, "register hand-over must balance");
  static_assert(kRegsLaunch * kThreads <= 65536, "launch registers");
  if (regs != kRegsLaunch) return cudaErrorInvalidConfiguration;
  const size_t smem = Smem<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(k_bwd_dq<D, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int n_items = p.B * p.N1 * p.Mq_t;
  int grid = p.num_sms;
  if (n_items < grid) grid = n_items;
  if (grid < 1) grid = 1;
  k_bwd_dq<D, DT><<<grid, kThreads, smem, st>>>(m.q, m.k, m.v, m.dout, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(const Plan& p, const BwdMaps& m, cudaStream_t st) {
  if (p.dtype == kDtBF16)
    return p.D == 128 ? launch_t<128, kDtBF16>(p, m, st) : launch_t<64, kDtBF16>(p, m, st);
  return p.D == 128 ? launch_t<128, kDtF16>(p, m, st) : launch_t<64, kDtF16>(p, m, st);
}

}  // namespace bsa
