// Split-KV forward for a few queries against a long key sequence (a decode
// step): per-chunk summaries, then a separate merge kernel.
//
// "Exact tiled softmax attention with block-recomputed vector-Jacobian
// products", Forward procedure: every row keeps a summary Sigma_i(I) of the key
// blocks seen so far and merges each new block's summary with the star rule.
// Here the key sequence is cut into `splits` contiguous chunks processed by
// different CTAs; each CTA runs the running-max recurrence of
// "txf-modern-flash-attention" (Hints) over its chunk in 32-key tiles and
// writes its summary (m, l, z) per query row (m in the exp2 domain,
// z = sum_j 2^(s_j - m) V_j unnormalised).  The merge kernel then combines the
// summaries of all chunks with the star rule,
//   M = max_s m_s,  l = sum_s 2^(m_s - M) l_s,  z = sum_s 2^(m_s - M) z_s,
// skipping empty summaries (m_s = -inf, the page's "bottom"), which is the
// same as folding the pairwise merge over the chunks in order (the merge is
// associative), and writes Y_i = z / l and L_i = ln 2 (M + log2 l).
//
// Queries sit at the end of the key sequence: query i is at absolute position
// i + nk - nq (causal: j <= i + nk - nq; window w: the w keys ending there;
// bit rows [nq][ceil(nk/32)]).
#include <math.h>

#include "common.cuh"

namespace exattn {
namespace {

constexpr int kTK = 32;       // keys per tile = one bitmask word
constexpr int kMaxNq = 64;

// 16-byte asynchronous global -> shared copies (cp.async), in commit groups.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Stage `valid` rows of a [rows][width] tile of T into shared memory rows of
// `ld_bytes` bytes (16-byte chunks, one warp); rows past `valid` are zeroed.
template <typename T>
__device__ __forceinline__ void stage_tile(uint8_t* dst, int ld_bytes, const T* src, int valid,
                                           int width) {
  const int chunks = width * static_cast<int>(sizeof(T)) / 16;
  const int lane = threadIdx.x & 31;
  for (int idx = lane; idx < kTK * chunks; idx += 32) {
    const int r = idx / chunks, c = idx - r * chunks;
    uint8_t* d = dst + r * ld_bytes + c * 16;
    if (r < valid)
      cp_async16(d, reinterpret_cast<const uint8_t*>(src + static_cast<size_t>(r) * width) + c * 16);
    else
      *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// 2^x with one MUFU operation (ex2.approx.ftz: relative error about 2^-22,
// 2^-inf = +0, which the empty-summary handling relies on).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T>
__device__ __forceinline__ float to_f(T x) {
  return Elem<T>::cvt(x);
}

// Star merge of the chunk summaries of one (slice, query) row by one warp.
// Lanes split the chunks for the maximum and the sum; for z each lane owns 4
// columns and walks the chunks with unconditional 16-byte loads (an empty
// chunk's z is all zeros and its factor 2^(m_s - M) is 0), the factor
// broadcast from the lane that computed it.  kCoherent reads through L2 only,
// for summaries written by other CTAs of the same launch.
template <bool kCoherent>
__device__ __forceinline__ float ld_sum(const float* p) {
  if constexpr (kCoherent) return __ldcg(p);
  else return *p;
}
template <bool kCoherent>
__device__ __forceinline__ float4 ld_sum4(const float* p) {
  if constexpr (kCoherent) return __ldcg(reinterpret_cast<const float4*>(p));
  else return *reinterpret_cast<const float4*>(p);
}

template <typename T, bool kCoherent>
__device__ void merge_row(const SplitArgs& a, int bh, int q, T* Y, float* L, unsigned* status) {
  const int lane = threadIdx.x & 31;
  const int S = a.splits, v = a.v;
  const size_t base = static_cast<size_t>(bh) * S * a.nq + q;  // row of chunk 0
  const size_t stride = a.nq;                                   // rows between chunks
  const size_t row = static_cast<size_t>(bh) * a.nq + q;
  float M = -INFINITY;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, ld_sum<kCoherent>(a.pm + base + s * stride));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
  T* yrow = Y + row * v;
  if (M == -INFINITY) {  // every chunk's summary is empty: the row's allowed set is empty
    for (int c = lane; c < v; c += 32) Elem<T>::store(yrow + c, 0.f);
    if (lane == 0) {
      L[row] = -INFINITY;
      raise_status(status, kStatusEmptyRow);
    }
    return;
  }
  float lsum = 0.f;
  for (int s = lane; s < S; s += 32) {
    const float ms = ld_sum<kCoherent>(a.pm + base + s * stride);
    if (ms != -INFINITY) lsum += fast_exp2(ms - M) * ld_sum<kCoherent>(a.pl + base + s * stride);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, o);
  const float inv = 1.f / lsum;
  for (int c0 = 4 * lane; c0 - 4 * lane < v; c0 += 128) {  // warp-uniform trip count
    const int cl = c0 < v ? c0 : 0;                          // lanes past v read column 0
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < S; s0 += 32) {
      float f_own = 0.f;
      if (s0 + lane < S) {
        const float ms = ld_sum<kCoherent>(a.pm + base + (s0 + lane) * stride);
        f_own = ms == -INFINITY ? 0.f : fast_exp2(ms - M);
      }
      const int cnt = min(32, S - s0);
#pragma unroll 8
      for (int k = 0; k < cnt; ++k) {
        const float f = __shfl_sync(0xFFFFFFFFu, f_own, k);
        const float4 z = ld_sum4<kCoherent>(a.pz + (base + (s0 + k) * stride) * v + cl);
        acc.x = fmaf(f, z.x, acc.x);
        acc.y = fmaf(f, z.y, acc.y);
        acc.z = fmaf(f, z.z, acc.z);
        acc.w = fmaf(f, z.w, acc.w);
      }
    }
    if (c0 < v) {
      Elem<T>::store(yrow + c0, acc.x * inv);
      Elem<T>::store(yrow + c0 + 1, acc.y * inv);
      Elem<T>::store(yrow + c0 + 2, acc.z * inv);
      Elem<T>::store(yrow + c0 + 3, acc.w * inv);
    }
  }
  if (lane == 0) L[row] = (M + log2f(lsum)) * kLn2;
}

// Separate merge pass (after splitkv_partial_kernel): one warp per row.
constexpr int kMergeThreads = 64;

template <typename T>
__global__ void __launch_bounds__(kMergeThreads) splitkv_merge_kernel(SplitArgs a, T* Y, float* L,
                                                                      unsigned* status) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (gw >= a.BH * a.nq) return;
  const int bh = gw / a.nq;
  merge_row<T, false>(a, bh, gw - bh * a.nq, Y, L, status);
}

// One warp per (batch*head, chunk): every query row of the chunk, lane = key
// of the current 32-key tile.  K and V tiles are double-buffered in shared
// memory (raw elements, rows padded by 16 bytes): tile t+1 streams in with
// cp.async while tile t is used.  Running (m, l) and z in shared memory.
template <typename T, int VPL>
__global__ void __launch_bounds__(32) splitkv_partial_kernel(SplitArgs a) {
  extern __shared__ __align__(16) uint8_t smraw[];
  const int d = a.d, v = a.v, nq = a.nq, nk = a.nk;
  const int kld = d * static_cast<int>(sizeof(T)) + 16;  // bytes per staged K row
  const int vld = v * static_cast<int>(sizeof(T)) + 16;
  float* Qs = reinterpret_cast<float*>(smraw);          // [nq][d]
  float* Zs = Qs + nq * d;                              // [nq][v]
  float* Ms = Zs + nq * v;                              // [nq]
  float* Ls = Ms + nq;                                  // [nq]
  uint8_t* stage = reinterpret_cast<uint8_t*>(Ls + nq + (4 - (2 * nq + nq * (d + v)) % 4) % 4);
  uint8_t* Kst[2] = {stage, stage + kTK * kld};
  uint8_t* Vst[2] = {stage + 2 * kTK * kld, stage + 2 * kTK * kld + kTK * vld};
  const int bh = blockIdx.y, split = blockIdx.x;
  const int lane = threadIdx.x;
  const int j_begin = split * a.chunk;
  const int j_end = min(nk, j_begin + a.chunk);
  const int off = nk - nq;
  const T* Qh = static_cast<const T*>(a.Q) + static_cast<size_t>(bh) * nq * d;
  const T* Kh = static_cast<const T*>(a.K) + static_cast<size_t>(bh) * nk * d;
  const T* Vh = static_cast<const T*>(a.V) + static_cast<size_t>(bh) * nk * v;

  for (int idx = lane; idx < nq * d; idx += 32) Qs[idx] = Elem<T>::load(Qh + idx);
  for (int idx = lane; idx < nq * v; idx += 32) Zs[idx] = 0.f;
  for (int q = lane; q < nq; q += 32) {
    Ms[q] = -INFINITY;
    Ls[q] = 0.f;
  }
  // First tile that any query can reach (window: the earliest query's window).
  int j_start = j_begin;
  if (a.mask_kind == kMaskWindow) j_start = max(j_start, (max(0, off - a.window + 1) / kTK) * kTK);

  if (j_start < j_end) {
    stage_tile(Kst[0], kld, Kh + static_cast<size_t>(j_start) * d, min(kTK, j_end - j_start), d);
    stage_tile(Vst[0], vld, Vh + static_cast<size_t>(j_start) * v, min(kTK, j_end - j_start), v);
  }
  cp_async_commit();
  int buf = 0;
  for (int j0 = j_start; j0 < j_end; j0 += kTK, buf ^= 1) {
    const int jn = j0 + kTK;
    if (jn < j_end) {  // prefetch the next tile into the other buffer
      stage_tile(Kst[buf ^ 1], kld, Kh + static_cast<size_t>(jn) * d, min(kTK, j_end - jn), d);
      stage_tile(Vst[buf ^ 1], vld, Vh + static_cast<size_t>(jn) * v, min(kTK, j_end - jn), v);
    }
    cp_async_commit();
    cp_async_wait<1>();  // the current tile has landed
    __syncwarp();
    const T* krow = reinterpret_cast<const T*>(Kst[buf] + lane * kld);
    const uint8_t* vt = Vst[buf];
    const int j = j0 + lane;
    for (int q = 0; q < nq; ++q) {
      const int ia = q + off;  // absolute position of query q
      bool ok = j < j_end;
      if (a.mask_kind == kMaskCausal) ok = ok && j <= ia;
      if (a.mask_kind == kMaskWindow) ok = ok && j <= ia && j > ia - a.window;
      if (a.mask_kind == kMaskBitmask && ok)
        ok = (__ldg(a.bits + static_cast<size_t>(q) * a.words_per_row + (j0 >> 5)) >> lane) & 1u;
      float s = -INFINITY;
      if (ok) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const float* qr = Qs + q * d;
        constexpr int E = 16 / sizeof(T);
        for (int e0 = 0; e0 < d; e0 += E) {
          const uint4 raw = *reinterpret_cast<const uint4*>(krow + e0);
          const T* ke = reinterpret_cast<const T*>(&raw);
#pragma unroll
          for (int k = 0; k < E; ++k) acc[k & 3] = fmaf(qr[e0 + k], to_f(ke[k]), acc[k & 3]);
        }
        s = ((acc[0] + acc[1]) + (acc[2] + acc[3])) * a.sl2;
      }
      float tmax = s;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xFFFFFFFFu, tmax, o));
      const float m_old = Ms[q];
      const float m_new = fmaxf(m_old, tmax);
      if (m_new == -INFINITY) continue;  // nothing allowed yet for this row (warp-uniform)
      const float alpha = m_old == -INFINITY ? 0.f : exp2f(m_old - m_new);
      const float p = ok ? exp2f(s - m_new) : 0.f;
      float psum = p;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xFFFFFFFFu, psum, o);
      const float l_new = Ls[q] * alpha + psum;
#pragma unroll
      for (int t = 0; t < VPL; ++t) {
        const int c = lane + 32 * t;
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 8
        for (int kk = 0; kk < kTK; kk += 2) {
          const float p0 = __shfl_sync(0xFFFFFFFFu, p, kk);
          const float p1 = __shfl_sync(0xFFFFFFFFu, p, kk + 1);
          if (c < v) {
            acc0 = fmaf(p0, to_f(reinterpret_cast<const T*>(vt + kk * vld)[c]), acc0);
            acc1 = fmaf(p1, to_f(reinterpret_cast<const T*>(vt + (kk + 1) * vld)[c]), acc1);
          }
        }
        if (c < v) Zs[q * v + c] = fmaf(Zs[q * v + c], alpha, acc0 + acc1);
      }
      __syncwarp();
      if (lane == 0) {
        Ms[q] = m_new;
        Ls[q] = l_new;
      }
      __syncwarp();
    }
    __syncwarp();  // every lane is done with this buffer before it is refilled
  }
  cp_async_wait<0>();
  // This chunk's summary of every query row.
  __syncwarp();
  for (int q = 0; q < nq; ++q) {
    const size_t row = (static_cast<size_t>(bh) * a.splits + split) * nq + q;
    if (lane == 0) {
      a.pm[row] = Ms[q];
      a.pl[row] = Ls[q];
    }
    for (int c = lane; c < v; c += 32) a.pz[row * v + c] = Zs[q * v + c];
  }
}

// ---------------------------------------------------------------------------
// Register-resident chunk kernel for nq <= 4 (the decode shapes).
//
// A group of G lanes covers one key row: lane gl of the group holds 16-byte
// pieces gl, gl + G, ... of the K and V rows (CPL pieces), so one warp-wide
// 16-byte load reads 32/G whole consecutive rows.  Each warp keeps U key
// steps of K and V in flight in registers, forms the scores by a partial dot
// product and a reduction inside the group, and runs the running-max
// recurrence per group.  At the end the groups of a warp, then the four warps
// of the CTA, are combined with the star merge into one summary per chunk.
// No key tile goes through shared memory.

template <typename T> struct Piece;
template <> struct Piece<float> {
  static constexpr int E = 4;
  __device__ static void unpack(const uint4& r, float (&f)[4]) {
    f[0] = __uint_as_float(r.x);
    f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z);
    f[3] = __uint_as_float(r.w);
  }
};
template <> struct Piece<__nv_bfloat16> {
  static constexpr int E = 8;
  // bf16 -> fp32 is exact: the 16 bits become the high half of the fp32 word.
  __device__ static void unpack(const uint4& r, float (&f)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

constexpr int kRegWarps = 4;
constexpr int kRegMaxNq = 4;

template <typename T, int G, int CPL, int NQ>
__global__ void __launch_bounds__(32 * kRegWarps) splitkv_reg_kernel(SplitArgs a) {
  constexpr int E = Piece<T>::E;
  constexpr int KPW = 32 / G;     // key rows per warp-wide load
  constexpr int U = (NQ == 1 ? 8 : 4) / CPL;  // key steps in flight
  constexpr int STEP = KPW * U;   // keys per warp iteration
  constexpr int W = CPL * E;      // elements of a row held by one lane
  __shared__ float red_m[kRegWarps][NQ], red_l[kRegWarps][NQ];
  __shared__ __align__(16) float red_z[kRegWarps][NQ][256];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane / G, gl = lane % G;
  const int d = a.d, v = a.v, nq = a.nq, nk = a.nk;
  const int kch = d / E, vch = v / E;  // 16-byte pieces per K / V row
  const int bh = blockIdx.y, split = blockIdx.x;
  const int j_begin = split * a.chunk;
  const int j_end = min(nk, j_begin + a.chunk);
  const int off = nk - nq;
  const T* Qh = static_cast<const T*>(a.Q) + static_cast<size_t>(bh) * nq * d;
  const T* Kh = static_cast<const T*>(a.K) + static_cast<size_t>(bh) * nk * d;
  const T* Vh = static_cast<const T*>(a.V) + static_cast<size_t>(bh) * nk * v;

  // Query slices, with c * log2(e) folded in so that scores are in the exp2 domain.
  float qf[NQ][W];
#pragma unroll
  for (int q = 0; q < NQ; ++q)
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int pc = gl + c * G;
      float f[E];
      if (q < nq && pc < kch) Piece<T>::unpack(*reinterpret_cast<const uint4*>(Qh + q * d + pc * E), f);
      else
#pragma unroll
        for (int e = 0; e < E; ++e) f[e] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) qf[q][c * E + e] = f[e] * a.sl2;
    }
  float m[NQ], l[NQ], z[NQ][W];
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    m[q] = -INFINITY;
    l[q] = 0.f;
#pragma unroll
    for (int e = 0; e < W; ++e) z[q][e] = 0.f;
  }

  int j_start = j_begin;
  if (a.mask_kind == kMaskWindow) j_start = max(j_start, off - a.window + 1);

  for (int j0 = j_start + warp * STEP; j0 < j_end; j0 += kRegWarps * STEP) {
    uint4 kr[U][CPL], vr[U][CPL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int key = j0 + u * KPW + g;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const int pc = gl + c * G;
        kr[u][c] = (key < j_end && pc < kch) ? ld_stream16(Kh + static_cast<size_t>(key) * d + pc * E)
                                             : make_uint4(0u, 0u, 0u, 0u);
        vr[u][c] = (key < j_end && pc < vch) ? ld_stream16(Vh + static_cast<size_t>(key) * v + pc * E)
                                             : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (q >= nq) break;  // warp-uniform
      const int ia = q + off;
      float s[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          float f[E];
          Piece<T>::unpack(kr[u][c], f);
#pragma unroll
          for (int e = 0; e < E; e += 2) {
            acc0 = fmaf(qf[q][c * E + e], f[e], acc0);
            acc1 = fmaf(qf[q][c * E + e + 1], f[e + 1], acc1);
          }
        }
        float part = acc0 + acc1;
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
        const int key = j0 + u * KPW + g;
        bool ok = key < j_end;
        if (a.mask_kind == kMaskCausal) ok = ok && key <= ia;
        if (a.mask_kind == kMaskWindow) ok = ok && key <= ia && key > ia - a.window;
        if (a.mask_kind == kMaskBitmask && ok)
          ok = (__ldg(a.bits + static_cast<size_t>(q) * a.words_per_row + (key >> 5)) >> (key & 31)) & 1u;
        s[u] = ok ? part : -INFINITY;
      }
      float mx = m[q];
#pragma unroll
      for (int u = 0; u < U; ++u) mx = fmaxf(mx, s[u]);
      // A group that has seen no allowed key keeps its empty state (ref = 0
      // makes every factor exp2(-inf) = 0 without producing NaN).
      const float ref = mx == -INFINITY ? 0.f : mx;
      const float alpha = fast_exp2(m[q] - ref);
      float psum = 0.f;
#pragma unroll
      for (int e = 0; e < W; ++e) z[q][e] *= alpha;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float p = fast_exp2(s[u] - ref);
        psum += p;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          float f[E];
          Piece<T>::unpack(vr[u][c], f);
#pragma unroll
          for (int e = 0; e < E; ++e) z[q][c * E + e] = fmaf(p, f[e], z[q][c * E + e]);
        }
      }
      l[q] = l[q] * alpha + psum;
      m[q] = mx;
    }
  }

  // Star merge of the groups of this warp (lanes with equal gl hold the same
  // columns, so xor offsets that are multiples of G pair matching slices).
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    float M = m[q];
#pragma unroll
    for (int o = G; o < 32; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    const float f = M == -INFINITY ? 0.f : fast_exp2(m[q] - M);
    float lq = l[q] * f;
#pragma unroll
    for (int o = G; o < 32; o <<= 1) lq += __shfl_xor_sync(0xFFFFFFFFu, lq, o);
#pragma unroll
    for (int e = 0; e < W; ++e) {
      float ze = z[q][e] * f;
#pragma unroll
      for (int o = G; o < 32; o <<= 1) ze += __shfl_xor_sync(0xFFFFFFFFu, ze, o);
      z[q][e] = ze;
    }
    if (q < nq && lane < G) {
      if (lane == 0) {
        red_m[warp][q] = M;
        red_l[warp][q] = lq;
      }
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const int pc = gl + c * G;
        if (pc < vch)
#pragma unroll
          for (int e = 0; e < E; ++e) red_z[warp][q][pc * E + e] = z[q][c * E + e];
      }
    }
  }
  __syncthreads();
  // Star merge of the warps; one summary per (bh, chunk, query).
  for (int idx = threadIdx.x; idx < nq * v; idx += 32 * kRegWarps) {
    const int q = idx / v, col = idx - q * v;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kRegWarps; ++w) M = fmaxf(M, red_m[w][q]);
    float zc = 0.f, lq = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kRegWarps; ++w) {
        const float f = fast_exp2(red_m[w][q] - M);
        zc = fmaf(f, red_z[w][q][col], zc);
        lq = fmaf(f, red_l[w][q], lq);
      }
    }
    const size_t row = (static_cast<size_t>(bh) * a.splits + split) * nq + q;
    a.pz[row * v + col] = zc;
    if (col == 0) {
      a.pm[row] = M;
      a.pl[row] = lq;
    }
  }
  // The last CTA of this slice to finish merges all of its chunk summaries
  // (each CTA publishes its summary with a fence before counting itself).
  __shared__ bool s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(a.counters + bh, 1u) == static_cast<unsigned>(a.splits - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (warp < nq) merge_row<T, true>(a, bh, warp, static_cast<T*>(a.Y), a.L, a.status);
}

template <typename T, int G, int CPL>
cudaError_t reg_launch(const SplitArgs& a, cudaStream_t s) {
  before_launch(kKernSplitPartial, s);
  if (a.nq == 1)
    splitkv_reg_kernel<T, G, CPL, 1><<<dim3(a.splits, a.BH), 32 * kRegWarps, 0, s>>>(a);
  else
    splitkv_reg_kernel<T, G, CPL, kRegMaxNq><<<dim3(a.splits, a.BH), 32 * kRegWarps, 0, s>>>(a);
  after_launch(kKernSplitPartial, s);
  return cudaGetLastError();
}

template <typename T>
cudaError_t reg_dispatch(const SplitArgs& a, cudaStream_t s) {
  const int pieces = max(a.d, a.v) * static_cast<int>(sizeof(T)) / 16;
  if (pieces <= 8) return reg_launch<T, 8, 1>(a, s);
  if (pieces <= 16) return reg_launch<T, 16, 1>(a, s);
  if constexpr (sizeof(T) == 2) {  // d, v <= 256 bf16 is at most 32 pieces
    return reg_launch<T, 32, 1>(a, s);
  } else {
    if (pieces <= 32) return reg_launch<T, 32, 1>(a, s);
    return reg_launch<T, 32, 2>(a, s);
  }
}

template <typename T, int VPL>
cudaError_t partial_launch(const SplitArgs& a, cudaStream_t s) {
  const size_t smem = splitkv_smem_bytes(a.nq, a.d, a.v, static_cast<int>(sizeof(T)));
  auto kern = splitkv_partial_kernel<T, VPL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  before_launch(kKernSplitPartial, s);
  kern<<<dim3(a.splits, a.BH), 32, smem, s>>>(a);
  after_launch(kKernSplitPartial, s);
  return cudaGetLastError();
}

template <typename T>
cudaError_t splitkv_launch_t(const SplitArgs& a, void* Y, float* L, unsigned* status,
                             cudaStream_t s) {
  if (a.nq <= kRegMaxNq) return reg_dispatch<T>(a, s);  // merges in its last CTA per slice
  cudaError_t e;
  if (a.v <= 32) e = partial_launch<T, 1>(a, s);
  else if (a.v <= 64) e = partial_launch<T, 2>(a, s);
  else if (a.v <= 128) e = partial_launch<T, 4>(a, s);
  else e = partial_launch<T, 8>(a, s);
  if (e != cudaSuccess) return e;
  const int rows = a.BH * a.nq;
  before_launch(kKernSplitMerge, s);
  splitkv_merge_kernel<T><<<(rows * 32 + kMergeThreads - 1) / kMergeThreads, kMergeThreads, 0,
                            s>>>(a, static_cast<T*>(Y), L, status);
  after_launch(kKernSplitMerge, s);
  return cudaGetLastError();
}

}  // namespace

size_t splitkv_smem_bytes(int nq, int d, int v, int elem_bytes) {
  // fp32 Q, z, m, l (padded to 16 bytes) + two staged K and two staged V
  // tiles of raw elements, each row padded by 16 bytes.
  const size_t f = static_cast<size_t>(nq) * (d + v) + 2 * static_cast<size_t>(nq);
  const size_t fbytes = (f + 3) / 4 * 4 * sizeof(float);
  return fbytes + 2 * kTK * (static_cast<size_t>(d) * elem_bytes + 16) +
         2 * kTK * (static_cast<size_t>(v) * elem_bytes + 16);
}

int splitkv_max_queries() { return kMaxNq; }
int splitkv_reg_max_queries() { return kRegMaxNq; }

cudaError_t launch_splitkv_merge(const SplitArgs& a, int dtype, void* Y, float* L,
                                 unsigned* status, cudaStream_t s) {
  const int rows = a.BH * a.nq;
  const unsigned blocks = (rows * 32 + kMergeThreads - 1) / kMergeThreads;
  before_launch(kKernSplitMerge, s);
  if (dtype == kF32)
    splitkv_merge_kernel<float><<<blocks, kMergeThreads, 0, s>>>(a, static_cast<float*>(Y), L,
                                                                 status);
  else
    splitkv_merge_kernel<__nv_bfloat16><<<blocks, kMergeThreads, 0, s>>>(
        a, static_cast<__nv_bfloat16*>(Y), L, status);
  after_launch(kKernSplitMerge, s);
  return cudaGetLastError();
}

cudaError_t launch_splitkv(const SplitArgs& a, int dtype, void* Y, float* L, unsigned* status,
                           cudaStream_t s) {
  return dtype == kF32 ? splitkv_launch_t<float>(a, Y, L, status, s)
                       : splitkv_launch_t<__nv_bfloat16>(a, Y, L, status, s);
}

}  // namespace exattn
