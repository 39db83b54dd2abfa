// Device-side helpers shared by every exattn kernel: the allowed-key predicate,
// element conversion and the device status word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace exattn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Bits of the device status word (first word of every workspace).
constexpr unsigned kStatusEmptyRow = 1u;
constexpr unsigned kStatusTimeout = 2u;

__device__ __forceinline__ void raise_status(unsigned* status, unsigned bit) {
  atomicOr(status, bit);
}

// Membership of key j in A_i ("Exact tiled softmax attention ...", Inputs),
// for 0 <= i, j < n.  Keys j >= n do not exist and are never allowed.
struct MaskView {
  int kind;
  int n;
  int window;
  int words_per_row;
  const uint32_t* bits;

  __device__ __forceinline__ bool allowed(int i, int j) const {
    if (j >= n || j < 0) return false;
    switch (kind) {
      case kMaskCausal: return j <= i;
      case kMaskWindow: return j <= i && j > i - window;
      case kMaskBitmask:
        return (__ldg(bits + (size_t)i * words_per_row + (j >> 5)) >> (j & 31)) & 1u;
      default: return true;
    }
  }
};

template <typename T> struct Elem;
// load(): read one element from GLOBAL memory; cvt(): convert a value already
// in registers.
template <> struct Elem<float> {
  static __device__ __forceinline__ float load(const float* p) { return __ldg(p); }
  static __device__ __forceinline__ float cvt(float x) { return x; }
  static __device__ __forceinline__ void store(float* p, float x) { *p = x; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
  }
  static __device__ __forceinline__ float cvt(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, float x) {
    *p = __float2bfloat16_rn(x);
  }
};

}  // namespace exattn
