// bsa_device.cuh - small device helpers shared by the tensor-core kernels:
// the 16-bit operand type of a run (bf16 or fp16) with its packing of two
// floats into one 32-bit word (low half = first value), and the error report
// a kernel writes into the workspace header when a bounded wait gives up.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bsa_common.h"

namespace bsa {

template <int DT>
struct Elem;
template <>
struct Elem<kDtBF16> {
  using T = __nv_bfloat16;
  static constexpr int kAB = 1;  // operand-type code of the tcgen05 instruction descriptor
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

// Bounds-check build (compiled with BSA_CHECKS=1): the work items and list
// entries the planner wrote are validated where the kernels read them, and an
// index outside its array is recorded (kErrBounds, the check's id in
// kHdrCheckWhere) and replaced by an empty item or entry, so that nothing
// reads or writes outside its array and nothing traps. In the default build
// the checks compile to nothing.
#if defined(BSA_CHECKS) && BSA_CHECKS
constexpr bool kChecks = true;
#else
constexpr bool kChecks = false;
#endif

// First failure wins the code word; every failing wait is counted by code.
__device__ __forceinline__ void record_error(int* header, int where) {
  atomicCAS(&header[kHdrErrorWhere], 0, where);
  atomicExch(&header[kHdrError], 1);
  atomicAdd(&header[kHdrErrorCounts + (where & 15)], 1);
}

__device__ __forceinline__ void check_failed(int* header, int id) {
  atomicCAS(&header[kHdrCheckWhere], 0, id);
  record_error(header, kErrBounds);
}

// A work item {key tile, entry begin, entry end, slot} as claimed (x < 0: end
// of work); out of range -> an empty item every role skips.
__device__ __forceinline__ int4 checked_item(const Plan& p, int4 it) {
  if (kChecks && it.x >= 0 &&
      !(it.x < p.NGC && it.y >= 0 && it.y <= it.z && it.z <= p.max_entries && it.w >= -1 &&
        it.w < p.max_slots)) {
    check_failed(p.header, kCheckItem);
    return make_int4(0, 0, 0, -1);
  }
  return it;
}

// Entry e of the work list; out of range -> query tile 0 of local head 0 with
// no sub-block selected, which contributes nothing.
__device__ __forceinline__ int32_t load_entry(const Plan& p, int e) {
  const int32_t ent = p.entries[e];
  if (kChecks && (entry_it(ent) >= p.Mq_t || entry_hl(ent) >= p.G)) {
    check_failed(p.header, kCheckEntry);
    return 0;
  }
  return ent;
}

}  // namespace bsa
