// SIMT fp32 kernels: the exact-fp32 path (fp32 inputs, or any shape the tensor
// core kernels do not take) and the two memory-bound helpers of the reverse
// pass (delta, dQ conversion).
//
// Forward: one CTA per (32 query rows, batch*head); key tiles of 32, online
// softmax in registers (exp2 of scores pre-multiplied by c*log2(e)), eight
// threads per query row.  Reverse: one CTA per (32 keys, batch*head); loops
// over query tiles, recomputes p from the frozen L, keeps dK and dV for its
// keys in registers and adds dQ contributions to an fp32 accumulator.
#include <math.h>

#include "common.cuh"

namespace exattn {
namespace {

constexpr int kBQ = 32;   // query rows per tile
constexpr int kBK = 32;   // keys per tile (one bitmask word per row)
constexpr int kThreads = 256;

// Range of key tiles [kt0, kt1) that can intersect A_i for rows [i0, i1]
// (absolute positions i + nk - n).
__device__ __forceinline__ void key_tile_range(const Problem& p, int i0, int i1, int& kt0,
                                               int& kt1) {
  const int off = p.nk - p.n;
  kt0 = 0;
  kt1 = (p.nk + kBK - 1) / kBK;
  if (p.mask_kind == kMaskCausal || p.mask_kind == kMaskWindow)
    kt1 = i1 + off < 0 ? 0 : min(kt1, (i1 + off) / kBK + 1);
  if (p.mask_kind == kMaskWindow) kt0 = max(0, i0 + off - p.window + 1) / kBK;
}

template <typename T>
__device__ __forceinline__ void load_tile(float* dst, int ld, const T* src, int row0, int rows,
                                          int n, int width) {
  for (int idx = threadIdx.x; idx < rows * width; idx += kThreads) {
    int r = idx / width, c = idx - r * width;
    int g = row0 + r;
    dst[r * ld + c] = g < n ? Elem<T>::load(src + (size_t)g * width + c) : 0.f;
  }
}

template <typename T, int VPT>
__global__ void __launch_bounds__(kThreads) simt_fwd_kernel(FwdArgs a) {
  const Problem p = a.p;
  const int n = p.n, nk = p.nk, d = p.d, v = p.v, dp = d + 1;
  extern __shared__ float smem[];
  float* Qs = smem;
  float* Ks = Qs + kBQ * dp;
  float* Vs = Ks + kBK * dp;
  float* Ps = Vs + kBK * v;

  const int bh = blockIdx.y, q0 = blockIdx.x * kBQ;
  const int tid = threadIdx.x, r = tid >> 3, l8 = tid & 7;
  const int i = q0 + r;
  const T* Qh = static_cast<const T*>(a.Q) + (size_t)bh * n * d;
  const T* Kh = static_cast<const T*>(a.K) + (size_t)bh * nk * d;
  const T* Vh = static_cast<const T*>(a.V) + (size_t)bh * nk * v;
  MaskView mask{p.mask_kind, nk, nk - n, p.window, p.words_per_row, p.bitmask};

  load_tile(Qs, dp, Qh, q0, kBQ, n, d);
  const float sl2 = p.scale * kLog2e;
  float m = -INFINITY, l = 0.f;
  float o[VPT];
#pragma unroll
  for (int t = 0; t < VPT; ++t) o[t] = 0.f;

  int kt0, kt1;
  key_tile_range(p, q0, min(q0 + kBQ, n) - 1, kt0, kt1);
  for (int kt = kt0; kt < kt1; ++kt) {
    const int j0 = kt * kBK;
    if (p.mask_kind == kMaskBitmask) {
      // Whole-tile skip: no row of this query tile allows a key of this tile.
      bool any = false;
      if (tid < kBQ && q0 + tid < n)
        any = __ldg(p.bitmask + (size_t)(q0 + tid) * p.words_per_row + (j0 >> 5)) != 0u;
      if (!__syncthreads_or(any)) continue;
    }
    __syncthreads();
    load_tile(Ks, dp, Kh, j0, kBK, nk, d);
    load_tile(Vs, v, Vh, j0, kBK, nk, v);
    __syncthreads();

    // Dropout keep bits of this row for the tile's four 8-key groups: lane l8 < 4
    // of the row draws group l8 (one Philox call), the row's lanes share them.
    uint32_t kbits = 0xFFFFFFFFu;
    if (p.drop_t != 0) {
      uint32_t mine = 0;
      if (l8 < 4 && i < n) mine = keep_byte(p.drop_t, p.seed_lo, p.seed_hi, bh, i, (j0 >> 3) + l8);
      kbits = 0;
#pragma unroll
      for (int t = 0; t < 4; ++t)
        kbits |= ((__shfl_sync(0xffffffffu, mine, (tid & 24) + t) >> l8) & 1u) << t;
    }
    float s[4];
    float tmax = -INFINITY;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int kc = l8 + 8 * t;
      float acc = 0.f;
      const float* qr = Qs + r * dp;
      const float* kr = Ks + kc * dp;
      #pragma unroll 4
        for (int e = 0; e < d; ++e) acc = fmaf(qr[e], kr[e], acc);
      s[t] = (i < n && mask.allowed(i, j0 + kc)) ? acc * sl2 : -INFINITY;
      tmax = fmaxf(tmax, s[t]);
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    const float mnew = fmaxf(m, tmax);
    const float mref = mnew == -INFINITY ? 0.f : mnew;
    const float alpha = m == -INFINITY ? 0.f : exp2f(m - mref);
    float psum = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float pv = exp2f(s[t] - mref);
      psum += pv;  // the row sum is of the undropped p
      Ps[r * (kBK + 1) + l8 + 8 * t] = ((kbits >> t) & 1u) ? pv : 0.f;
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
    l = l * alpha + psum;
    m = mnew;
    __syncwarp();
#pragma unroll
    for (int t = 0; t < VPT; ++t) {
      const int col = l8 + 8 * t;
      if (col < v) {
        float acc = o[t] * alpha;
        #pragma unroll 4
        for (int k = 0; k < kBK; ++k) acc = fmaf(Ps[r * (kBK + 1) + k], Vs[k * v + col], acc);
        o[t] = acc;
      }
    }
  }

  if (i < n) {
    T* Yr = static_cast<T*>(a.Y) + ((size_t)bh * n + i) * v;
    const float inv = l > 0.f ? p.drop_scale / l : 0.f;
#pragma unroll
    for (int t = 0; t < VPT; ++t) {
      const int col = l8 + 8 * t;
      if (col < v) Elem<T>::store(Yr + col, o[t] * inv);
    }
    if (l8 == 0) {
      a.L[(size_t)bh * n + i] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
      if (!(l > 0.f)) raise_status(a.status, kStatusEmptyRow);
    }
  }
}

template <typename T, int DPT, int VPT>
__global__ void __launch_bounds__(kThreads) simt_bwd_kernel(BwdArgs a) {
  const Problem p = a.p;
  const int n = p.n, nk = p.nk, d = p.d, v = p.v, dp = d + 1, vp = v + 1;
  const int off = nk - n;
  extern __shared__ float smem[];
  float* Ks = smem;
  float* Vs = Ks + kBK * dp;
  float* Qs = Vs + kBK * vp;
  float* dYs = Qs + kBQ * dp;
  float* Pt = dYs + kBQ * vp;
  float* dSt = Pt + kBK * (kBQ + 1);
  float* Ls = dSt + kBK * (kBQ + 1);
  float* Ds = Ls + kBQ;

  __shared__ uint8_t kbits_s[kBQ][4];  // dropout keep bits of the current query tile
  const int bh = blockIdx.y, j0 = blockIdx.x * kBK;
  const int tid = threadIdx.x, r = tid >> 3, l8 = tid & 7;
  const int j = j0 + r;
  const T* Qh = static_cast<const T*>(a.Q) + (size_t)bh * n * d;
  const T* Kh = static_cast<const T*>(a.K) + (size_t)bh * nk * d;
  const T* Vh = static_cast<const T*>(a.V) + (size_t)bh * nk * v;
  const T* dYh = static_cast<const T*>(a.dY) + (size_t)bh * n * v;
  const float* Lh = a.L + (size_t)bh * n;
  const float* Dh = a.delta + (size_t)bh * a.npad;
  float* dQh = a.dQacc + (size_t)bh * n * d;
  MaskView mask{p.mask_kind, nk, off, p.window, p.words_per_row, p.bitmask};
  const float c = p.scale, sl2 = p.scale * kLog2e;

  load_tile(Ks, dp, Kh, j0, kBK, nk, d);
  load_tile(Vs, vp, Vh, j0, kBK, nk, v);
  float dk[DPT], dv[VPT];
#pragma unroll
  for (int t = 0; t < DPT; ++t) dk[t] = 0.f;
#pragma unroll
  for (int t = 0; t < VPT; ++t) dv[t] = 0.f;

  // Query tiles whose rows can allow a key of [j0, j1] (row i is at i + off).
  const int j1 = min(j0 + kBK, nk) - 1;
  int qt0 = 0, qt1 = (n + kBQ - 1) / kBQ;
  if (p.mask_kind == kMaskCausal || p.mask_kind == kMaskWindow) qt0 = max(0, j0 - off) / kBQ;
  if (p.mask_kind == kMaskWindow) {
    const int last = j1 - off + p.window - 1;  // last row whose window reaches j1
    qt1 = last < 0 ? 0 : min(qt1, last / kBQ + 1);
  }

  for (int qt = qt0; qt < qt1; ++qt) {
    const int q0 = qt * kBQ;
    if (p.mask_kind == kMaskBitmask) {
      bool any = false;
      if (tid < kBQ && q0 + tid < n)
        any = __ldg(p.bitmask + (size_t)(q0 + tid) * p.words_per_row + (j0 >> 5)) != 0u;
      if (!__syncthreads_or(any)) continue;
    }
    __syncthreads();
    load_tile(Qs, dp, Qh, q0, kBQ, n, d);
    load_tile(dYs, vp, dYh, q0, kBQ, n, v);
    if (p.drop_t != 0 && tid < kBQ * 4) {  // keep bits: 32 queries x four 8-key groups
      const int qq = tid >> 2, g = tid & 3, gi = q0 + qq;
      kbits_s[qq][g] = gi < n ? static_cast<uint8_t>(keep_byte(p.drop_t, p.seed_lo, p.seed_hi,
                                                               bh, gi, (j0 >> 3) + g))
                              : 0;
    }
    if (tid < kBQ) {
      const int gi = q0 + tid;
      Ls[tid] = gi < n ? Lh[gi] * kLog2e : -INFINITY;
      Ds[tid] = gi < n ? Dh[gi] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int qc = l8 + 8 * t, gi = q0 + qc;
      float pv = 0.f, ds = 0.f;
      if (gi < n && j < nk && Ls[qc] != -INFINITY && mask.allowed(gi, j)) {
        float acc = 0.f;
        #pragma unroll 4
        for (int e = 0; e < d; ++e) acc = fmaf(Ks[r * dp + e], Qs[qc * dp + e], acc);
        pv = exp2f(acc * sl2 - Ls[qc]);
        float dpv = 0.f;
        #pragma unroll 4
        for (int e = 0; e < v; ++e) dpv = fmaf(Vs[r * vp + e], dYs[qc * vp + e], dpv);
        if (p.drop_t != 0) {
          // Replayed mask: dV takes p xi s, and dP = xi s (G_i . V_j).
          const float xs = ((kbits_s[qc][r >> 3] >> (r & 7)) & 1u) ? p.drop_scale : 0.f;
          ds = pv * (dpv * xs - Ds[qc]);
          pv *= xs;
        } else {
          ds = pv * (dpv - Ds[qc]);
        }
      }
      Pt[r * (kBQ + 1) + qc] = pv;
      dSt[r * (kBQ + 1) + qc] = ds;
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < VPT; ++t) {
      const int col = l8 + 8 * t;
      if (col < v) {
        float acc = dv[t];
        #pragma unroll 4
        for (int q = 0; q < kBQ; ++q) acc = fmaf(Pt[r * (kBQ + 1) + q], dYs[q * vp + col], acc);
        dv[t] = acc;
      }
    }
#pragma unroll
    for (int t = 0; t < DPT; ++t) {
      const int col = l8 + 8 * t;
      if (col < d) {
        float acc = dk[t];
        #pragma unroll 4
        for (int q = 0; q < kBQ; ++q) acc = fmaf(dSt[r * (kBQ + 1) + q], Qs[q * dp + col], acc);
        dk[t] = acc;
      }
    }
    // dQ rows of this query tile: thread (query r, columns l8 + 8t).
    const int gi = q0 + r;
    if (gi < n) {
#pragma unroll
      for (int t = 0; t < DPT; ++t) {
        const int col = l8 + 8 * t;
        if (col < d) {
          float acc = 0.f;
          #pragma unroll 4
          for (int k = 0; k < kBK; ++k) acc = fmaf(dSt[k * (kBQ + 1) + r], Ks[k * dp + col], acc);
          atomicAdd(dQh + (size_t)gi * d + col, c * acc);
        }
      }
    }
  }

  if (j < nk) {
    T* dKr = static_cast<T*>(a.dK) + ((size_t)bh * nk + j) * d;
    T* dVr = static_cast<T*>(a.dV) + ((size_t)bh * nk + j) * v;
#pragma unroll
    for (int t = 0; t < DPT; ++t)
      if (l8 + 8 * t < d) Elem<T>::store(dKr + l8 + 8 * t, c * dk[t]);
#pragma unroll
    for (int t = 0; t < VPT; ++t)
      if (l8 + 8 * t < v) Elem<T>::store(dVr + l8 + 8 * t, dv[t]);
  }
}

// delta_i = sum_a dY_ia Y_ia and lse2_i = L_i log2(e) over padded rows
// [BH][npad]: one row per group of G lanes, 16-byte loads.  Padding rows
// (i >= n) get delta = 0 and lse2 = +inf, as do rows with L_i = -inf (an empty
// allowed set), so that exp2(s - lse2) = 0 there.
struct DeltaArgs {
  const void* Y;
  const void* dY;
  const float* L;
  float* delta;
  float* lse2;
  int n, npad, v;
  size_t rows;  // BH * npad
  unsigned* status;  // EMPTY_ROW when a row's L is -inf (its allowed set was empty)
};

__device__ __forceinline__ void delta_store(const DeltaArgs& a, size_t row, float acc) {
  const size_t bh = row / a.npad;
  const int i = static_cast<int>(row - bh * a.npad);
  if (i < a.n) {
    const float L = a.L[bh * a.n + i];
    a.delta[row] = acc;
    a.lse2[row] = L == -INFINITY ? INFINITY : L * kLog2e;
    if (L == -INFINITY) raise_status(a.status, kStatusEmptyRow);
  } else {
    a.delta[row] = 0.f;
    a.lse2[row] = INFINITY;
  }
}

// One row per group of G lanes (G = v / elements per 16-byte vector, so each
// lane reads one vector of Y and one of dY per row); a grid-stride loop over
// rows with kRows rows in flight per group.  The trip count is the same for
// every lane, so the group reductions run converged.
constexpr int kDeltaRows = 4;

template <typename T, int G>
__global__ void __launch_bounds__(256, 4) delta_vec_kernel(DeltaArgs a) {
  constexpr int E = 16 / sizeof(T);  // elements per 16-byte vector
  constexpr int R = kDeltaRows;
  const int lane = static_cast<int>(threadIdx.x % G);
  const size_t groups = static_cast<size_t>(gridDim.x) * (256 / G);
  const size_t group = static_cast<size_t>(blockIdx.x) * (256 / G) + threadIdx.x / G;
  const size_t iters = (a.rows + groups * R - 1) / (groups * R);
  for (size_t it = 0; it < iters; ++it) {
    const size_t r0 = (it * groups + group) * R;
    uint4 va[R], vb[R];
    bool live[R];
    float Lr[R];  // L of row u, loaded (with Y and dY) by the lane that stores row u
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const size_t row = r0 + u;
      const size_t bh = row / a.npad;
      const int i = static_cast<int>(row - bh * a.npad);
      live[u] = row < a.rows && i < a.n;
      Lr[u] = -INFINITY;
      if (live[u]) {
        const size_t src = (bh * a.n + i) * a.v;
        va[u] = __ldcs(reinterpret_cast<const uint4*>(static_cast<const T*>(a.Y) + src) + lane);
        vb[u] = __ldcs(reinterpret_cast<const uint4*>(static_cast<const T*>(a.dY) + src) + lane);
        if (lane == u % G) Lr[u] = __ldcs(a.L + bh * a.n + i);
      }
    }
#pragma unroll
    for (int u = 0; u < R; ++u) {
      float acc = 0.f;
      if (live[u]) {
        const T* ea = reinterpret_cast<const T*>(&va[u]);
        const T* eb = reinterpret_cast<const T*>(&vb[u]);
#pragma unroll
        for (int e = 0; e < E; ++e) acc = fmaf(Elem<T>::cvt(ea[e]), Elem<T>::cvt(eb[e]), acc);
      }
#pragma unroll
      for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      // Padding rows (i >= n): delta 0, L log2(e) = +inf (p = 0 in the reverse kernels).
      if (r0 + u < a.rows && lane == u % G) {
        a.delta[r0 + u] = live[u] ? acc : 0.f;
        a.lse2[r0 + u] = live[u] && Lr[u] != -INFINITY ? Lr[u] * kLog2e : INFINITY;
        if (live[u] && Lr[u] == -INFINITY) raise_status(a.status, kStatusEmptyRow);
      }
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) delta_scalar_kernel(DeltaArgs a) {
  const size_t row = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  if (row < a.rows) {
    const size_t bh = row / a.npad;
    const int i = static_cast<int>(row - bh * a.npad);
    if (i < a.n) {
      const T* y = static_cast<const T*>(a.Y) + (bh * a.n + i) * a.v;
      const T* g = static_cast<const T*>(a.dY) + (bh * a.n + i) * a.v;
      for (int k = lane; k < a.v; k += 32) acc = fmaf(Elem<T>::load(y + k), Elem<T>::load(g + k), acc);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < a.rows && lane == 0) delta_store(a, row, acc);
}

template <typename T>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc,
                                                         T* __restrict__ out, size_t count) {
  for (size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x; k < count;
       k += (size_t)gridDim.x * blockDim.x)
    Elem<T>::store(out + k, acc[k]);
}

int per_thread(int width) { return width <= 64 ? 8 : width <= 128 ? 16 : 32; }

template <typename T, int VPT>
cudaError_t fwd_launch_t(const FwdArgs& a, cudaStream_t s) {
  const Problem& p = a.p;
  size_t smem = sizeof(float) * (size_t)(kBQ * (p.d + 1) + kBK * (p.d + 1) + kBK * p.v +
                                         kBQ * (kBK + 1));
  auto kern = simt_fwd_kernel<T, VPT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.n + kBQ - 1) / kBQ, p.BH);
  before_launch(kKernFwd, s);
  kern<<<grid, kThreads, smem, s>>>(a);
  after_launch(kKernFwd, s);
  return cudaGetLastError();
}

template <typename T, int DPT, int VPT>
cudaError_t bwd_launch_t(const BwdArgs& a, cudaStream_t s) {
  const Problem& p = a.p;
  size_t smem = sizeof(float) * (size_t)(kBK * (p.d + 1) + kBK * (p.v + 1) + kBQ * (p.d + 1) +
                                         kBQ * (p.v + 1) + 2 * kBK * (kBQ + 1) + 2 * kBQ);
  auto kern = simt_bwd_kernel<T, DPT, VPT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.nk + kBK - 1) / kBK, p.BH);
  before_launch(kKernBwd, s);
  kern<<<grid, kThreads, smem, s>>>(a);
  after_launch(kKernBwd, s);
  return cudaGetLastError();
}

template <typename T>
cudaError_t fwd_dispatch(const FwdArgs& a, cudaStream_t s) {
  switch (per_thread(a.p.v)) {
    case 8: return fwd_launch_t<T, 8>(a, s);
    case 16: return fwd_launch_t<T, 16>(a, s);
    default: return fwd_launch_t<T, 32>(a, s);
  }
}

template <typename T>
cudaError_t bwd_dispatch(const BwdArgs& a, cudaStream_t s) {
  // One register-array width for both d and v keeps the instantiation count small.
  switch (per_thread(a.p.d > a.p.v ? a.p.d : a.p.v)) {
    case 8: return bwd_launch_t<T, 8, 8>(a, s);
    case 16: return bwd_launch_t<T, 16, 16>(a, s);
    default: return bwd_launch_t<T, 32, 32>(a, s);
  }
}

template <typename T>
cudaError_t delta_dispatch(const BwdArgs& a, cudaStream_t s) {
  const Problem& p = a.p;
  DeltaArgs d{a.Y, a.dY, a.L, a.delta, a.lse2, p.n, a.npad, p.v, (size_t)p.BH * a.npad,
              a.status};
  constexpr int E = 16 / sizeof(T);
  const int vecs = p.v / E;
  before_launch(kKernDelta, s);
  if (p.v % E == 0 && (vecs & (vecs - 1)) == 0 && vecs <= 32) {
    // G lanes per row, one 16-byte vector per lane per row; one wave of as
    // many CTAs as fit on every SM (fewer when there are fewer rows).
    const int G = vecs;
    auto launch = [&](auto kern) {
      int dev = 0, sms = 148, per_sm = 4;
      if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0) != cudaSuccess ||
          per_sm < 1)
        per_sm = 1;
      const size_t need = (d.rows * G + 255) / 256;
      const size_t wave = static_cast<size_t>(sms) * per_sm;
      kern<<<static_cast<unsigned>(need < wave ? need : wave), 256, 0, s>>>(d);
    };
    switch (G) {
      case 1: launch(delta_vec_kernel<T, 1>); break;
      case 2: launch(delta_vec_kernel<T, 2>); break;
      case 4: launch(delta_vec_kernel<T, 4>); break;
      case 8: launch(delta_vec_kernel<T, 8>); break;
      case 16: launch(delta_vec_kernel<T, 16>); break;
      default: launch(delta_vec_kernel<T, 32>); break;
    }
  } else {
    const unsigned blocks = (unsigned)((d.rows * 32 + 255) / 256);
    delta_scalar_kernel<T><<<blocks, 256, 0, s>>>(d);
  }
  after_launch(kKernDelta, s);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_fwd(const FwdArgs& a, cudaStream_t s) {
  return a.p.dtype == kF32 ? fwd_dispatch<float>(a, s) : fwd_dispatch<__nv_bfloat16>(a, s);
}

cudaError_t launch_simt_bwd(const BwdArgs& a, cudaStream_t s) {
  if (simt_bwd_rt_supported(a.p)) return launch_simt_bwd_rt(a, s);
  return a.p.dtype == kF32 ? bwd_dispatch<float>(a, s) : bwd_dispatch<__nv_bfloat16>(a, s);
}

cudaError_t launch_delta(const BwdArgs& a, cudaStream_t s) {
  return a.p.dtype == kF32 ? delta_dispatch<float>(a, s) : delta_dispatch<__nv_bfloat16>(a, s);
}

cudaError_t launch_dq_convert(const BwdArgs& a, cudaStream_t s) {
  const size_t count = (size_t)a.p.BH * a.p.n * a.p.d;
  const unsigned blocks = (unsigned)((count + 255) / 256 < 152 * 64 ? (count + 255) / 256 : 152 * 64);
  before_launch(kKernDqConvert, s);
  if (a.p.dtype == kF32)
    dq_convert_kernel<float><<<blocks, 256, 0, s>>>(a.dQacc, static_cast<float*>(a.dQ), count);
  else
    dq_convert_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
        a.dQacc, static_cast<__nv_bfloat16*>(a.dQ), count);
  after_launch(kKernDqConvert, s);
  return cudaGetLastError();
}

}  // namespace exattn
