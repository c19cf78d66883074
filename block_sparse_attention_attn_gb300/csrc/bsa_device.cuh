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

// First failure wins the code word; every failing wait is counted by code.
__device__ __forceinline__ void record_error(int* header, int where) {
  atomicCAS(&header[kHdrErrorWhere], 0, where);
  atomicExch(&header[kHdrError], 1);
  atomicAdd(&header[kHdrErrorCounts + (where & 15)], 1);
}

}  // namespace bsa
