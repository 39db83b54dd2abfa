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
// for query row i and key j < nk; query i sits at absolute position i + off
// (off = nk - nq).  Keys j >= nk do not exist and are never allowed.
struct MaskView {
  int kind;
  int nk;
  int off;
  int window;
  int words_per_row;
  const uint32_t* bits;

  __device__ __forceinline__ bool allowed(int i, int j) const {
    if (j >= nk || j < 0) return false;
    const int a = i + off;
    switch (kind) {
      case kMaskCausal: return j <= a;
      case kMaskWindow: return j <= a && j > a - window;
      case kMaskBitmask:
        return (__ldg(bits + (size_t)i * words_per_row + (j >> 5)) >> (j & 31)) & 1u;
      default: return true;
    }
  }
};

// Philox-4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC 2011): each round multiplies counter words
// 0 and 2 by the round multipliers (keeping both 32-bit halves of the
// products), mixes the high halves into words 1 and 3 with the key, and the
// key advances by the Weyl increments between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t m0 = static_cast<uint64_t>(c.x) * 0xD2511F53u;  // one wide multiply each
    const uint64_t m1 = static_cast<uint64_t>(c.z) * 0xCD9E8D57u;
    const uint32_t lo0 = static_cast<uint32_t>(m0), hi0 = static_cast<uint32_t>(m0 >> 32);
    const uint32_t lo1 = static_cast<uint32_t>(m1), hi1 = static_cast<uint32_t>(m1 >> 32);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// Dropout keep bits of keys 8*jb .. 8*jb+7 of row i in slice bh: bit t is set
// when key 8*jb + t is kept.  Counter (jb, i, bh, 0), key (seed low, seed
// high); key 8*jb + t reads half t%2 of output word t/2 (low half first) and
// is kept when that 16-bit value is >= drop_t ("Exact tiled softmax attention
// with block-recomputed vector-Jacobian products", Reverse procedure: the
// reverse pass replays exactly these decisions).
__device__ __forceinline__ uint32_t keep_byte(uint32_t drop_t, uint32_t seed_lo, uint32_t seed_hi,
                                              int bh, int i, int jb) {
  const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(jb), static_cast<uint32_t>(i),
                                           static_cast<uint32_t>(bh), 0u),
                                seed_lo, seed_hi);
  const uint32_t th = drop_t << 16;  // word >= t * 2^16  <=>  high half >= t
  return static_cast<uint32_t>((w.x & 0xFFFFu) >= drop_t) |
         (static_cast<uint32_t>(w.x >= th) << 1) |
         (static_cast<uint32_t>((w.y & 0xFFFFu) >= drop_t) << 2) |
         (static_cast<uint32_t>(w.y >= th) << 3) |
         (static_cast<uint32_t>((w.z & 0xFFFFu) >= drop_t) << 4) |
         (static_cast<uint32_t>(w.z >= th) << 5) |
         (static_cast<uint32_t>((w.w & 0xFFFFu) >= drop_t) << 6) |
         (static_cast<uint32_t>(w.w >= th) << 7);
}

// The raw Philox words of keys 8*jb .. 8*jb+7 of row i in slice bh (key 8*jb + t
// reads half t%2 of word t/2; see keep_byte).
__device__ __forceinline__ uint4 keep_words(uint32_t seed_lo, uint32_t seed_hi, int bh, int i,
                                            int jb) {
  return philox4x32_10(make_uint4(static_cast<uint32_t>(jb), static_cast<uint32_t>(i),
                                  static_cast<uint32_t>(bh), 0u),
                       seed_lo, seed_hi);
}

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
