// bsa_fwd.cu - companion block-sparse attention forward on the sm_103a tensor
// cores: Out = softmax(scale * Q K^T over the selected blocks) V and
// softmaxLse = natural-log logsumexp of the selected scaled scores
// (aclnnBlockSparseAttentionGrad page, section 计算公式, forward part), with
// the online rescaling of the FlashAttentionScore page (section 实现原理): the
// running row max m and sum l are updated per key tile and the partial PV
// product is rescaled by exp(m_old - m_new) when the max grows.
//
// One persistent CTA per SM, 384 threads:
//   warp 8      producer: scans the mask row(s) of its query tile for selected
//               key tiles and streams K/V tiles through a 3-stage TMA ring;
//   warp 9      MMA issuer of S = Q K^T (into one of two TMEM buffers, as soon
//               as the P of tile m-2 in that buffer has been read) and TMEM
//               owner;
//   warp 10     MMA issuer of O_wg += P_wg V_wg (P read from TMEM), per
//               warpgroup as soon as its P is ready. Two issuers, because an
//               issuing thread blocks while the tensor pipe's queue is full:
//               with one, the PV product of tile m-1 waited behind the issue
//               of S(m), and so did S(m+1), which needs that PV's S buffer;
//   warps 0-7   softmax, two warpgroups: TMEM lane s = query row s, warpgroup
//               wg owns keys [64 wg, 64 wg + 64) of every tile and runs its
//               own online softmax over them (its own running max and sum)
//               into its own O accumulator O_wg += P_wg V_wg (a K = 64
//               product), so the two warpgroups never wait for each other
//               within an item; at the end of an item they swap their maxima
//               and sums through shared memory and each writes half of the
//               output columns from O_0 and O_1 rescaled to the common max.
//               The live keys of a tile (length, window, sub-block, token
//               mask) are one bit word per 32 columns.
// The rescale is lazy: O_wg is only rescaled when its row max grows by more
// than 8 (log2 units), so P stays below 2^8 and most tiles skip the TMEM
// round trip.
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
constexpr int kMmaWarp = 9;   // S = Q K^T; TMEM owner
constexpr int kPvWarp = 10;   // O += P V; warp 11 only lends its registers
// Registers per thread after the hand-over (launch: 384 x 168): the control
// warpgroup (warps 8-11) keeps 64, the two softmax warpgroups get 208 each
// (2 x 208 + 64 <= 3 x 168). Each budget has its own copy of the out-of-line
// wait loop (wait tags).
constexpr int kRegsLaunch = 168, kRegsCtl = 64, kRegsSoftmax = 208;
constexpr int kTagCtl = 1, kTagSoftmax = 2;
constexpr int kPanel = 128 * 128;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;  // O_wg at kColO + wg * D
constexpr float kRescaleThreshold = 8.f;
constexpr int kStages = 3;  // K/V ring depth

enum Bar {
  kQFull = 0, kQEmpty,
  kKvFull0, kKvFull1, kKvFull2, kKvEmpty0, kKvEmpty1, kKvEmpty2, kKvAux0, kKvAux1, kKvAux2,
  kSFull0, kSFull1,
  kPReady00, kPReady01, kPReady10, kPReady11,  // [S buffer][warpgroup]
  kPvDone00, kPvDone01, kPvDone10, kPvDone11,  // [S buffer][warpgroup]
  kOFull, kOEmpty, kXch0, kXch1,
  kItemFull0, kItemFull1, kItemEmpty0, kItemEmpty1,
  kDrain, kDrain2,
  kNumBars
};

template <int D>
struct Smem {
  static constexpr int kTileBytes = (D / 64) * kPanel;
  static constexpr int oQ = 0;
  static constexpr int oK = oQ + kTileBytes;             // [kStages]
  static constexpr int oV = oK + kStages * kTileBytes;   // [kStages]
  static constexpr int oXch = oV + kStages * kTileBytes;  // float [2][2][128] partial row maxima / sums
  static constexpr int oBar = oXch + 2048;
  static constexpr int oMisc = (oBar + kNumBars * 8 + 63) / 64 * 64;  // int4 slots need 16 B
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

// Packed fp32 pairs (two lanes of one 64-bit register) and three-input
// min / max: one instruction for two elements of the softmax loops.
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
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

struct FItem {
  int b, h, it;
};

__device__ __forceinline__ FItem decode(const Plan& p, int idx) {
  FItem r;
  r.it = idx % p.Mq_t;
  const int bh = idx / p.Mq_t;
  r.h = bh % p.N1;
  r.b = bh / p.N1;
  return r;
}

// Sub-block bits of key tile jt for query tile `it` of (b, h): selected,
// inside the valid range and meeting the sliding window.
__device__ __forceinline__ int fwd_tile_bits(const Plan& p, int b, int h, int it, int jt, int Lq,
                                             int Lk) {
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
    k_fwd(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
          const __grid_constant__ CUtensorMap tm_v, const FwdPlan f) {
  using S = Smem<D>;
  using E = Elem<DT>;
  using T = typename E::T;
  const Plan& p = f.p;
  constexpr int kPanels = D / 64;
  constexpr uint32_t kIdS = idesc_f16(128, 128, E::kAB, 0, 0);  // S = Q K^T
  constexpr uint32_t kIdO = idesc_f16(128, D, E::kAB, 0, 1);     // O += P V (A in TMEM)

  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::oBar);
  int* misc = reinterpret_cast<int*>(smem + S::oMisc);
  volatile int* abort_flag = misc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 1);
  int* item_slot = misc + 2;   // [2]
  int* meta = misc + 4;        // [kStages] per stage: jt | bits << 24, -1 = end of item
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(p.header, kErrSmemAlign);
    return;
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(&bars[kQFull], 1);
    mbar_init(&bars[kQEmpty], 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars[kKvFull0 + i], 1);
      mbar_init(&bars[kKvEmpty0 + i], 2 + kSoftmaxWarps);  // both MMA warps + softmax warps
      mbar_init(&bars[kKvAux0 + i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars[kPReady00 + i], kSoftmaxWarps / 2);  // the warps of one warpgroup
      mbar_init(&bars[kPvDone00 + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kSFull0 + i], 1);
      mbar_init(&bars[kXch0 + i], 32 * kSoftmaxWarps);  // every softmax thread posts a value
      mbar_init(&bars[kItemFull0 + i], 1);
      mbar_init(&bars[kItemEmpty0 + i], 2 + kSoftmaxWarps);
    }
    mbar_init(&bars[kOFull], 1);
    mbar_init(&bars[kOEmpty], kSoftmaxWarps);
    mbar_init(&bars[kDrain], 1);
    mbar_init(&bars[kDrain2], 1);
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  uint8_t* sQ = smem + S::oQ;
  uint8_t* sK0 = smem + S::oK;
  uint8_t* sV0 = smem + S::oV;

  if (warp >= kProdWarp) {
  regs_release<kRegsCtl>();  // all four warps of the control warpgroup
  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    uint32_t n = 0, itc = 0, aux[kStages] = {0u, 0u, 0u};
    bool ok = true;
    int pend_q = 0, pend_kv[kStages] = {0, 0, 0}, pend_aux[kStages] = {0, 0, 0};
    uint32_t par_kv[kStages] = {0u, 0u, 0u};
    while (ok) {
      const int slot = itc & 1;
      if (!mbar_wait<kTagCtl>(&bars[kItemEmpty0 + slot], ((itc >> 1) & 1) ^ 1, abort_flag)) {
        record_error(p.header, kErrWaitItem);
        break;
      }
      if (lane == 0) {
        const int idx = atomicAdd(&p.header[kHdrWorkCounter], 1);
        item_slot[slot] = idx < f.n_rows_items ? idx : -1;
        mbar_arrive(&bars[kItemFull0 + slot]);
      }
      __syncwarp();
      const int idx = item_slot[slot];
      if (idx < 0) break;
      const FItem fi = decode(p, idx);
      const int Lq = p.lq[fi.b], Lk = p.lk[fi.b];
      const int q0 = fi.it * 128;
      const bool has_rows = q0 < Lq;
      if (!mbar_wait<kTagCtl>(&bars[kQEmpty], (itc & 1) ^ 1, abort_flag)) {
        record_error(p.header, kErrWaitQ);
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[kQFull], S::kTileBytes);
        const int c1 = p.layout == kLayoutBNSD ? q0 : fi.h;
        const int c2 = p.layout == kLayoutBNSD ? fi.b * p.N1 + fi.h : p.cu_q[fi.b] + q0;
        for (int pn = 0; pn < kPanels; ++pn) tma_load_3d(sQ + pn * kPanel, &tm_q, &bars[kQFull], pn * 64, c1, c2);
      }
      pend_q = 1;
      const int ncolt = has_rows ? (Lk + 127) / 128 : 0;
      for (int jt0 = 0; jt0 < ncolt && ok; jt0 += 32) {
        const int jt = jt0 + lane;
        const int bits = jt < ncolt ? fwd_tile_bits(p, fi.b, fi.h, fi.it, jt, Lq, Lk) : 0;
        unsigned ball = __ballot_sync(0xffffffffu, bits != 0);
        while (ball && ok) {
          const int src = __ffs(ball) - 1;
          ball &= ball - 1;
          const int jsel = jt0 + src;
          const int bsel = __shfl_sync(0xffffffffu, bits, src);
          const int st = n % kStages;
          if (!mbar_wait<kTagCtl>(&bars[kKvEmpty0 + st], ((n / kStages) & 1) ^ 1, abort_flag)) {
            record_error(p.header, kErrWaitKV);
            ok = false;
            break;
          }
          const bool tail = (Lk - jsel * 128) < 128;
          uint8_t* sK = sK0 + st * S::kTileBytes;
          uint8_t* sV = sV0 + st * S::kTileBytes;
          if (lane == 0) {
            meta[st] = jsel | (bsel << 24);
            uint64_t* tb = tail ? &bars[kKvAux0 + st] : &bars[kKvFull0 + st];
            mbar_arrive_expect_tx(tb, 2 * S::kTileBytes);
            const int c1 = p.layout == kLayoutBNSD ? jsel * 128 : fi.h / p.G;
            const int c2 = p.layout == kLayoutBNSD ? fi.b * p.N2 + fi.h / p.G : p.cu_k[fi.b] + jsel * 128;
            for (int pn = 0; pn < kPanels; ++pn) {
              tma_load_3d(sK + pn * kPanel, &tm_k, tb, pn * 64, c1, c2);
              tma_load_3d(sV + pn * kPanel, &tm_v, tb, pn * 64, c1, c2);
            }
          }
          pend_kv[st] = tail ? 0 : 1;
          par_kv[st] = (n / kStages) & 1;
          if (tail) {
            pend_aux[st] = 1;
            if (!mbar_wait<kTagCtl>(&bars[kKvAux0 + st], aux[st] & 1, abort_flag)) {
              record_error(p.header, kErrWaitKV);
              ok = false;
              break;
            }
            aux[st]++;
            pend_aux[st] = 0;
            zero_rows(sV, kPanels, Lk - jsel * 128, lane);  // 0 * NaN padding would poison O
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kKvFull0 + st]);
          }
          ++n;
        }
      }
      if (!ok) break;
      // end-of-item marker
      const int st = n % kStages;
      if (!mbar_wait<kTagCtl>(&bars[kKvEmpty0 + st], ((n / kStages) & 1) ^ 1, abort_flag)) {
        record_error(p.header, kErrWaitKV);
        break;
      }
      if (lane == 0) {
        meta[st] = -1;
        mbar_arrive(&bars[kKvFull0 + st]);
      }
      __syncwarp();
      ++n;
      ++itc;
    }
    if (*abort_flag) {
      if (pend_q) mbar_wait_drain(&bars[kQFull], (itc & 1));
      for (int st = 0; st < kStages; ++st) {
        if (pend_kv[st]) mbar_wait_drain(&bars[kKvFull0 + st], par_kv[st]);
        if (pend_aux[st]) mbar_wait_drain(&bars[kKvAux0 + st], aux[st] & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------ MMA issuer: S
    uint32_t n = 0, itc = 0;  // n: K/V stages (end markers included)
    uint32_t m = 0;           // m: computed key tiles (S/P buffers)
    int where = 0;
    const uint32_t aQ = smem_u32(sQ);
    while (true) {
      const int slot = itc & 1;
      if (!mbar_wait<kTagCtl>(&bars[kItemFull0 + slot], (itc >> 1) & 1, abort_flag)) { where = kErrWaitItem; break; }
      const int idx = item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + slot]);
      if (idx < 0) break;
      if (!mbar_wait<kTagCtl>(&bars[kQFull], itc & 1, abort_flag)) { where = kErrWaitQ; break; }
      tc_fence_after();
      while (true) {
        const int st = n % kStages;
        if (!mbar_wait<kTagCtl>(&bars[kKvFull0 + st], (n / kStages) & 1, abort_flag)) { where = kErrWaitKV; break; }
        const int mt = meta[st];
        __syncwarp();
        if (mt < 0) {
          if (lane == 0) mbar_arrive(&bars[kKvEmpty0 + st]);
          ++n;
          break;
        }
        // S(m) into buffer m & 1 once both PV halves of tile m-2 have read its P
        const uint32_t sb = m & 1;
        if (!mbar_wait<kTagCtl>(&bars[kPvDone00 + 2 * sb], ((m >> 1) & 1) ^ 1, abort_flag) ||
            !mbar_wait<kTagCtl>(&bars[kPvDone00 + 2 * sb + 1], ((m >> 1) & 1) ^ 1, abort_flag)) {
          where = kErrWaitMisc;
          break;
        }
        tc_fence_after();
        const uint32_t aK = smem_u32(sK0 + st * S::kTileBytes);
        const uint32_t colS = sb ? kColS1 : kColS0;
        if (lane == 0) {
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * kPanel + (k & 3) * 32;
            mma_ss(tmem + colS, sdesc_sw128(aQ + off, 16, 1024), sdesc_sw128(aK + off, 16, 1024), kIdS, k > 0);
          }
          tc_commit(&bars[kSFull0 + sb]);
          tc_commit(&bars[kKvEmpty0 + st]);  // K of the stage read
        }
        __syncwarp();
        ++n;
        ++m;
      }
      if (where) break;
      if (lane == 0) tc_commit(&bars[kQEmpty]);  // the item's last S has read Q
      __syncwarp();
      ++itc;
    }
    if (where) record_error(p.header, where);
    if (*abort_flag) {
      if (lane == 0) tc_commit(&bars[kDrain]);
      __syncwarp();
      mbar_wait_drain(&bars[kDrain], 0);
    }
  } else if (warp == kPvWarp) {
    // --------------------------------------------------- MMA issuer: P V
    uint32_t n = 0, itc = 0, m = 0;  // as in the S issuer
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
        const int st = n % kStages;
        if (!mbar_wait<kTagCtl>(&bars[kKvFull0 + st], (n / kStages) & 1, abort_flag)) { where = kErrWaitKV; break; }
        const int mt = meta[st];
        __syncwarp();
        if (mt < 0) {
          if (lane == 0) mbar_arrive(&bars[kKvEmpty0 + st]);
          ++n;
          break;
        }
        // O_wg += P_wg(m) V_wg for both warpgroups, each as soon as its P is
        // ready: A = P_wg (TMEM, packed over the warpgroup's S columns of
        // buffer m & 1), B = rows [64 wg, 64 wg + 64) of V of stage st
        // (MN-major); the item's first product starts the accumulators
        const uint32_t colS = (m & 1) ? kColS1 : kColS0;
        const uint32_t aV = smem_u32(sV0 + st * S::kTileBytes);
        for (int wg = 0; wg < 2 && !where; ++wg) {
          if (!mbar_wait<kTagCtl>(&bars[kPReady00 + 2 * (m & 1) + wg], (m >> 1) & 1, abort_flag)) {
            where = kErrWaitP;
            break;
          }
          if (j == 0 && wg == 0 && !mbar_wait<kTagCtl>(&bars[kOEmpty], (itc & 1) ^ 1, abort_flag)) {
            where = kErrWaitAcc;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ts(tmem + kColO + wg * D, tmem + colS + 64 * wg + 8 * k,
                     sdesc_sw128(aV + (4 * wg + k) * 2048, kPanel, 1024), kIdO,
                     (j == 0 && k == 0) ? 0u : 1u);
            tc_commit(&bars[kPvDone00 + 2 * (m & 1) + wg]);
            if (wg == 1) tc_commit(&bars[kKvEmpty0 + st]);  // V of the stage read
          }
          __syncwarp();
        }
        if (where) break;
        ++j;
        ++n;
        ++m;
      }
      if (where) break;
      // every item waits for the previous epilogue exactly once (a parity
      // wait cannot tell phase c from phase c-2, so no item may skip it)
      if (j == 0 && !mbar_wait<kTagCtl>(&bars[kOEmpty], (itc & 1) ^ 1, abort_flag)) {
        where = kErrWaitAcc;
        break;
      }
      if (lane == 0) tc_commit(&bars[kOFull]);
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
    // ------------------------------------------------------------- softmax
    const int qd = warp & 3, wg = warp >> 2;
    const int s = qd * 32 + lane;  // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    float* xch = reinterpret_cast<float*>(smem + S::oXch);
    uint32_t n = 0, itc = 0, m_step = 0;  // stages / computed key tiles (as in the MMA warp)
    uint32_t xs = 0;                       // exchanges through xch (maxima per tile, sums per item)
    int where = 0;
    while (true) {
      const int slot = itc & 1;
      if (!mbar_wait<kTagSoftmax>(&bars[kItemFull0 + slot], (itc >> 1) & 1, abort_flag)) { where = kErrWaitItem; break; }
      const int idx = item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + slot]);
      if (idx < 0) break;
      const FItem fi = decode(p, idx);
      const int Lq = p.lq[fi.b], Lk = p.lk[fi.b];
      const bool s_ok = fi.it * 128 + s < Lq;
      float m = -INFINITY, l = 0.f;  // running max (log2 units) and this warpgroup's sum
      int j = 0;
      while (true) {
        const int st = n % kStages;
        if (!mbar_wait<kTagSoftmax>(&bars[kKvFull0 + st], (n / kStages) & 1, abort_flag)) { where = kErrWaitKV; break; }
        const int mt = meta[st];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kKvEmpty0 + st]);
        if (mt < 0) { ++n; break; }
        const int jt = mt & 0xFFFFFF, bits = mt >> 24;
        const uint32_t sb = m_step & 1;
        const uint32_t colS = sb ? kColS1 : kColS0;
        if (!mbar_wait<kTagSoftmax>(&bars[kSFull0 + sb], (m_step >> 1) & 1, abort_flag)) { where = kErrWaitS; break; }
        tc_fence_after();
        // live columns: inside the key length and the sliding window ([t_lo,
        // t_hi)), in a selected key sub-block, kept by the token mask;
        // live_bits(c) has bit k set when key 32c + k of the tile takes part
        int t_lo = 0, t_hi = Lk - jt * 128;
        if (p.win) {
          const int2 w = win_span((int64_t)fi.it * 128 + s, (int64_t)jt * 128, -p.win_pre, p.win_next);
          t_lo = w.x;
          t_hi = min(t_hi, w.y);
        }
        const uint32_t* amr = p.am ? p.am_row + (int64_t)(fi.it * 128 + s) * p.am_wk + 4 * jt : nullptr;
        const int s_sub = p.rb == 2 ? (s >> 6) : 0;
        auto live_bits = [&](int c) -> uint32_t {
          const int t_sub = p.cb == 2 ? (c >> 1) : 0;
          if (!(s_ok && ((bits >> (s_sub * 2 + t_sub)) & 1))) return 0u;
          const uint32_t b = bit_range(t_lo - 32 * c, t_hi - 32 * c);
          return amr != nullptr ? b & ~amr[c] : b;
        };
        // this warpgroup's 64 keys of the tile, read once
        uint32_t x[64];
        tmem_ld64(tmem + lane_off + colS + 64 * wg, x);
        const uint32_t live0 = live_bits(2 * wg), live1 = live_bits(2 * wg + 1);
        // every key of the half takes part (the common case): no per-key tests
        const bool all_live = (live0 & live1) == 0xFFFFFFFFu;
        float mx;
        {
          // the max of the raw scores, scaled once (a negative scale turns it
          // into the min)
          const bool pos = p.scale_log2 >= 0.f;
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          if (all_live && pos) {
#pragma unroll
            for (int k = 0; k < 64; k += 2)
              m4[(k >> 1) & 3] = max3(m4[(k >> 1) & 3], __uint_as_float(x[k]), __uint_as_float(x[k + 1]));
          } else if (all_live) {
            float n4[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
#pragma unroll
            for (int k = 0; k < 64; k += 2)
              n4[(k >> 1) & 3] = min3(n4[(k >> 1) & 3], __uint_as_float(x[k]), __uint_as_float(x[k + 1]));
#pragma unroll
            for (int i = 0; i < 4; ++i) m4[i] = -n4[i];
          } else {
#pragma unroll
            for (int k = 0; k < 64; ++k) {
              const uint32_t lv = k < 32 ? live0 : live1;
              const float v = pos ? __uint_as_float(x[k]) : -__uint_as_float(x[k]);
              m4[k & 3] = fmaxf(m4[k & 3], ((lv >> (k & 31)) & 1u) ? v : -INFINITY);
            }
          }
          const float mr = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          mx = mr == -INFINITY ? -INFINITY : (pos ? mr : -mr) * p.scale_log2;
        }
        const bool grow = mx > m + kRescaleThreshold || (m == -INFINITY && mx > -INFINITY);
        // O rows of this warpgroup whose max grows are rescaled by alpha (after
        // the P of this tile is computed, so the scores are no longer live)
        const float alpha = (grow && m != -INFINITY) ? ex2_approx(m - mx) : 1.f;
        if (grow) {
          l = (m == -INFINITY) ? 0.f : l * alpha;
          m = mx;
        }
        float rs4[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[32];
        if (all_live) {
          // pairs of keys: one packed FMA for both exponents, one packed add
          // into two running pair sums
          const uint64_t c2 = f2(__float_as_uint(p.scale_log2), __float_as_uint(p.scale_log2));
          const uint64_t nm2 = f2(__float_as_uint(-m), __float_as_uint(-m));
          uint64_t sA = 0ull, sB = 0ull;
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            float t0, t1;
            f2split(fma2(f2(x[2 * k], x[2 * k + 1]), c2, nm2), t0, t1);
            const float e0 = ex2_approx(t0);
            const float e1 = ex2_approx(t1);
            const uint64_t e = f2(__float_as_uint(e0), __float_as_uint(e1));
            if (k & 1) sB = add2(sB, e);
            else sA = add2(sA, e);
            pk[k] = E::pack(e0, e1);
          }
          f2split(sA, rs4[0], rs4[1]);
          f2split(sB, rs4[2], rs4[3]);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const uint32_t lv = k < 16 ? live0 : live1;
            const int b0 = (2 * k) & 31;
            const float e0 = ex2_approx(fmaf(__uint_as_float(x[2 * k]), p.scale_log2, -m));
            const float e1 = ex2_approx(fmaf(__uint_as_float(x[2 * k + 1]), p.scale_log2, -m));
            const float p0 = ((lv >> b0) & 1u) ? e0 : 0.f;
            const float p1 = ((lv >> (b0 + 1)) & 1u) ? e1 : 0.f;
            rs4[k & 3] += p0 + p1;
            pk[k] = E::pack(p0, p1);
          }
        }
        const float rs = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
        if (__any_sync(0xffffffffu, grow) && j > 0) {
          // after this warpgroup's previous PV product has landed
          const uint32_t pb = (m_step - 1) & 1;
          if (!mbar_wait<kTagSoftmax>(&bars[kPvDone00 + 2 * pb + wg], ((m_step - 1) >> 1) & 1, abort_flag)) {
            where = kErrWaitMisc;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + kColO + wg * D + 32 * c, o);
            if (alpha != 1.f) {
#pragma unroll
              for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            }
            tmem_st32(tmem + lane_off + kColO + wg * D + 32 * c, o);
          }
        }
        // P packed in place over the first half of this warpgroup's S columns
        tmem_st32(tmem + lane_off + colS + 64 * wg, pk);
        l += rs;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kPReady00 + 2 * sb + wg]);
        ++j;
        ++n;
        ++m_step;
      }
      if (where) break;
      // epilogue: the common max M = max(m_0, m_1) and sum L = sum_wg l_wg 2^(m_wg - M)
      // (two exchanges through shared memory), Out = sum_wg O_wg 2^(m_wg - M) / L,
      // lse = (M + log2 L) * ln 2; warpgroup wg writes columns [wg D/2, wg D/2 + D/2)
      float m_o;
      {
        float* xb = xch + (xs & 1) * 256;
        xb[wg * 128 + s] = m;
        mbar_arrive(&bars[kXch0 + (xs & 1)]);
        if (!mbar_wait<kTagSoftmax>(&bars[kXch0 + (xs & 1)], (xs >> 1) & 1, abort_flag)) { where = kErrWaitMisc; break; }
        m_o = xb[(wg ^ 1) * 128 + s];
        ++xs;
      }
      const float M = fmaxf(m, m_o);
      const float a_own = M == -INFINITY ? 0.f : ex2_approx(m - M);
      const float a_oth = M == -INFINITY ? 0.f : ex2_approx(m_o - M);
      {
        float* lb = xch + (xs & 1) * 256;
        lb[wg * 128 + s] = l * a_own;
        mbar_arrive(&bars[kXch0 + (xs & 1)]);
        if (!mbar_wait<kTagSoftmax>(&bars[kXch0 + (xs & 1)], (xs >> 1) & 1, abort_flag)) { where = kErrWaitMisc; break; }
        l = l * a_own + lb[(wg ^ 1) * 128 + s];
        ++xs;
      }
      m = M;
      if (!mbar_wait<kTagSoftmax>(&bars[kOFull], itc & 1, abort_flag)) { where = kErrWaitAcc; break; }
      tc_fence_after();
      const int srow = fi.it * 128 + s;
      const bool write_row = p.layout == kLayoutBNSD ? (srow < p.Sq) : (srow < Lq);
      const bool live = s_ok && l > 0.f;
      const float inv = live ? 1.f / l : 0.f;
      // weights of O_0 and O_1 for this row
      const float w0 = (wg == 0 ? a_own : a_oth) * inv, w1 = (wg == 0 ? a_oth : a_own) * inv;
      int64_t ooff;
      int64_t sd;
      if (p.layout == kLayoutBNSD) {
        ooff = fi.b * f.out_st[0] + fi.h * f.out_st[1] + (int64_t)srow * f.out_st[2];
        sd = f.out_st[3];
      } else {
        ooff = ((int64_t)p.cu_q[fi.b] + srow) * f.out_st[0] + fi.h * f.out_st[1];
        sd = f.out_st[2];
      }
      T* out = static_cast<T*>(f.out) + ooff;
#pragma unroll 1
      for (int c = wg * (D / 64); c < (wg + 1) * (D / 64); ++c) {
        uint32_t o0[32], o1[32];
        if (j > 0) {
          tmem_ld32(tmem + lane_off + kColO + 32 * c, o0);
          tmem_ld32(tmem + lane_off + kColO + D + 32 * c, o1);
        }
        if (write_row) {
          // combined row values, kept in o0
#pragma unroll
          for (int k = 0; k < 32; ++k)
            o0[k] = __float_as_uint((live && j > 0)
                                        ? __uint_as_float(o0[k]) * w0 + __uint_as_float(o1[k]) * w1
                                        : 0.f);
          if (f.out_vec) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 u;
              u.x = E::pack(__uint_as_float(o0[8 * q]), __uint_as_float(o0[8 * q + 1]));
              u.y = E::pack(__uint_as_float(o0[8 * q + 2]), __uint_as_float(o0[8 * q + 3]));
              u.z = E::pack(__uint_as_float(o0[8 * q + 4]), __uint_as_float(o0[8 * q + 5]));
              u.w = E::pack(__uint_as_float(o0[8 * q + 6]), __uint_as_float(o0[8 * q + 7]));
              *reinterpret_cast<uint4*>(out + 32 * c + 8 * q) = u;
            }
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const uint32_t pk = E::pack(__uint_as_float(o0[k]), 0.f);
              out[(32 * c + k) * sd] = *reinterpret_cast<const T*>(&pk);
            }
          }
        }
      }
      if (write_row && wg == 0) {
        int64_t li;
        if (p.layout == kLayoutBNSD)
          li = ((int64_t)fi.b * p.N1 + fi.h) * p.Sq + srow;
        else
          li = ((int64_t)p.cu_q[fi.b] + srow) * p.N1 + fi.h;
        f.lse_out[li] = live ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kOEmpty]);
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
cudaError_t launch_t(const FwdPlan& f, const FwdMaps& m, cudaStream_t st) {
  const size_t smem = Smem<D>::kBytes;
  // The register hand-over only balances when every thread starts with
  // kRegsLaunch registers (a claim beyond what the others release would wait
  // for registers nobody frees).
  static const int regs = [] {
    cudaFuncAttributes fa{};
    return cudaFuncGetAttributes(&fa, k_fwd<D, DT>) == cudaSuccess ? fa.numRegs : -1;
  }();
  static_assert(2 * kRegsSoftmax + kRegsCtl <= 3 * kRegsLaunch, "register hand-over must balance");
  static_assert(kRegsLaunch * kThreads <= 65536, "launch registers");
  if (regs != kRegsLaunch) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(k_fwd<D, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int grid = f.p.num_sms;
  if (f.n_rows_items < grid) grid = f.n_rows_items;
  if (grid < 1) grid = 1;
  k_fwd<D, DT><<<grid, kThreads, smem, st>>>(m.q, m.k, m.v, f);
  return cudaGetLastError();
}

}  // namespace

size_t fwd_smem_bytes(int D) { return D == 128 ? Smem<128>::kBytes : Smem<64>::kBytes; }

cudaError_t launch_fwd(const FwdPlan& f, const FwdMaps& m, cudaStream_t st) {
  if (f.p.dtype == kDtBF16)
    return f.p.D == 128 ? launch_t<128, kDtBF16>(f, m, st) : launch_t<64, kDtBF16>(f, m, st);
  return f.p.D == 128 ? launch_t<128, kDtF16>(f, m, st) : launch_t<64, kDtF16>(f, m, st);
}

}  // namespace bsa
