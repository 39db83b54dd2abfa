// Register-tiled SIMT reverse pass (fp32 arithmetic) for d, v <= 128.  Widths
// other than 64 and 128 (multiples of 4) run on the kernel of width 64 or 128:
// rows are loaded with their own widths and zero-filled, and only the true
// columns are stored.
//
// The Reverse procedure of "Exact tiled softmax attention with block-
// recomputed vector-Jacobian products": per key block, for every query tile
// that can reach it, recompute p_ij = exp(s_ij - L_i) from Q, K and the frozen
// L, form gamma_ij = p_ij (G_i . V_j - delta_i), and accumulate
//   dV_j += p_ij G_i,   dK_j += c gamma_ij Q_i,   dQ_i += c gamma_ij K_j.
// delta_i = G_i . Y_i comes from the delta kernel (HarshvardhanJ/
// FlashAttention, backward section).  With dropout, p in dV and the G_i . V_j
// factor carry the replayed keep mask and scale.
//
// One CTA = 64 keys of one (batch, head), 256 threads; it loops over query
// tiles of 32.  Thread (ty, tx) = (tid / 16, tid % 16) owns keys 4ty..4ty+3:
//   S, dP:  a 4 x 2 block (queries 2tx, 2tx+1), operands from transposed tiles
//           (K^T, V^T resident; Q^T, dY^T per tile) as float4 / float2 loads;
//   dV, dK: 4 x (V/16) and 4 x (D/16) accumulators in registers, columns
//           4tx..4tx+3 (+64), operands P^T, dS^T and the row-major Q, dY tiles;
//   dQ:     queries 2ty, 2ty+1 x the same columns, from dS and row-major K,
//           added to the fp32 accumulator with 16-byte vector reductions.
// Every inner-loop shared-memory load is a broadcast or a conflict-free vector
// load, so the loops run at about one load per four to eight FMAs.
#include <math.h>

#include "common.cuh"

namespace exattn {
namespace {

constexpr int kBK = 64;  // keys per CTA
constexpr int kBQ = 32;  // queries per tile
constexpr int kThreads = 256;

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

template <int D, int V>
struct RtLayout {
  static constexpr int LK = kBK + 4;  // row stride of the [width][64] transposed tiles
  static constexpr int LQ = kBQ + 4;  // row stride of the [width][32] transposed tiles
  static constexpr int KT = 0;                    // K^T [D][LK]
  static constexpr int VT = KT + D * LK;          // V^T [V][LK]
  static constexpr int KS = VT + V * LK;          // K   [64][D + 4]
  static constexpr int QT = KS + kBK * (D + 4);   // Q^T [D][LQ]
  static constexpr int QS = QT + D * LQ;          // Q   [32][D + 4]
  static constexpr int YT = QS + kBQ * (D + 4);   // dY^T [V][LQ]
  static constexpr int YS = YT + V * LQ;          // dY  [32][V + 4]
  static constexpr int PT = YS + kBQ * (V + 4);   // (p xi s)^T [32][LK]
  static constexpr int ST = PT + kBQ * LK;        // dS^T [32][LK]
  static constexpr int SS = ST + kBQ * LK;        // dS   [64][LQ]
  static constexpr int LV = SS + kBK * LQ;        // L log2(e) of the tile [32]
  static constexpr int DV = LV + kBQ;             // delta of the tile [32]
  static constexpr int FLOATS = DV + kBQ;
};

template <typename T, int D, int V>
__global__ void __launch_bounds__(kThreads, 1) simt_bwd_rt_kernel(BwdArgs a) {
  using Lay = RtLayout<D, V>;
  constexpr int LK = Lay::LK, LQ = Lay::LQ;
  constexpr int CD = D / 64, CV = V / 64;  // float4 column groups per thread (0-63, 64-127)
  extern __shared__ __align__(16) float sm[];
  float* Kt = sm + Lay::KT;
  float* Vt = sm + Lay::VT;
  float* Ks = sm + Lay::KS;
  float* Qt = sm + Lay::QT;
  float* Qs = sm + Lay::QS;
  float* Yt = sm + Lay::YT;
  float* Ys = sm + Lay::YS;
  float* Pt = sm + Lay::PT;
  float* St = sm + Lay::ST;
  float* Ss = sm + Lay::SS;
  float* Lv = sm + Lay::LV;
  float* Dv = sm + Lay::DV;

  const Problem p = a.p;
  const int n = p.n, nk = p.nk, off = nk - n;
  const int bh = blockIdx.y, j0 = blockIdx.x * kBK;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int dw = p.d, vw = p.v;  // widths in memory (<= D, V)
  const T* Qh = static_cast<const T*>(a.Q) + (size_t)bh * n * dw;
  const T* Kh = static_cast<const T*>(a.K) + (size_t)bh * nk * dw;
  const T* Vh = static_cast<const T*>(a.V) + (size_t)bh * nk * vw;
  const T* Yh = static_cast<const T*>(a.dY) + (size_t)bh * n * vw;
  const float* Lh = a.lse2 + (size_t)bh * a.npad;
  const float* Dh = a.delta + (size_t)bh * a.npad;
  float* dQh = a.dQacc + (size_t)bh * n * dw;
  MaskView mask{p.mask_kind, nk, off, p.window, p.words_per_row, p.bitmask};
  const float c = p.scale, sl2 = p.scale * kLog2e;

  // K, V of the block: transposed (S, dP operands) and K row-major (dQ operand).
  for (int idx = tid; idx < kBK * D; idx += kThreads) {
    const int r = idx / D, col = idx - r * D, g = j0 + r;
    const float x = g < nk && col < dw ? Elem<T>::load(Kh + (size_t)g * dw + col) : 0.f;
    Kt[col * LK + r] = x;
    Ks[r * (D + 4) + col] = x;
  }
  for (int idx = tid; idx < kBK * V; idx += kThreads) {
    const int r = idx / V, col = idx - r * V, g = j0 + r;
    Vt[col * LK + r] = g < nk && col < vw ? Elem<T>::load(Vh + (size_t)g * vw + col) : 0.f;
  }

  float dv[4][4 * CV], dk[4][4 * CD];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
#pragma unroll
    for (int e = 0; e < 4 * CV; ++e) dv[r][e] = 0.f;
#pragma unroll
    for (int e = 0; e < 4 * CD; ++e) dk[r][e] = 0.f;
  }

  // Query tiles whose rows can reach a key of [j0, j1] (row i sits at i + off).
  const int j1 = min(j0 + kBK, nk) - 1;
  int qt0 = 0, qt1 = (n + kBQ - 1) / kBQ;
  if (p.mask_kind == kMaskCausal || p.mask_kind == kMaskWindow) qt0 = max(0, j0 - off) / kBQ;
  if (p.mask_kind == kMaskWindow) {
    const int last = j1 - off + p.window - 1;
    qt1 = last < 0 ? 0 : min(qt1, last / kBQ + 1);
  }

  for (int qt = qt0; qt < qt1; ++qt) {
    const int q0 = qt * kBQ;
    if (p.mask_kind == kMaskBitmask) {
      // Whole-tile skip: no row of the query tile allows a key of the block.
      bool any = false;
      if (tid < kBQ && q0 + tid < n) {
        const uint32_t* row = p.bitmask + (size_t)(q0 + tid) * p.words_per_row;
        const int w0 = j0 >> 5;
        any = __ldg(row + w0) != 0u || (w0 + 1 < p.words_per_row && __ldg(row + w0 + 1) != 0u);
      }
      if (!__syncthreads_or(any)) continue;
    }
    __syncthreads();  // the previous tile's operands are no longer read
    for (int idx = tid; idx < kBQ * D; idx += kThreads) {
      const int r = idx / D, col = idx - r * D, g = q0 + r;
      const float x = g < n && col < dw ? Elem<T>::load(Qh + (size_t)g * dw + col) : 0.f;
      Qt[col * LQ + r] = x;
      Qs[r * (D + 4) + col] = x;
    }
    for (int idx = tid; idx < kBQ * V; idx += kThreads) {
      const int r = idx / V, col = idx - r * V, g = q0 + r;
      const float x = g < n && col < vw ? Elem<T>::load(Yh + (size_t)g * vw + col) : 0.f;
      Yt[col * LQ + r] = x;
      Ys[r * (V + 4) + col] = x;
    }
    if (tid < kBQ) {
      Lv[tid] = Lh[q0 + tid];  // +inf on padding and empty rows: p = 0 there
      Dv[tid] = Dh[q0 + tid];
    }
    __syncthreads();

    // S and dP: keys 4ty..4ty+3 x queries 2tx, 2tx+1.
    float s[4][2], dp[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) s[r][0] = s[r][1] = dp[r][0] = dp[r][1] = 0.f;
#pragma unroll 8
    for (int e = 0; e < D; ++e) {
      const float4 k4 = *reinterpret_cast<const float4*>(Kt + e * LK + 4 * ty);
      const float2 q2 = *reinterpret_cast<const float2*>(Qt + e * LQ + 2 * tx);
      const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        s[r][0] = fmaf(kk[r], q2.x, s[r][0]);
        s[r][1] = fmaf(kk[r], q2.y, s[r][1]);
      }
    }
#pragma unroll 8
    for (int e = 0; e < V; ++e) {
      const float4 v4 = *reinterpret_cast<const float4*>(Vt + e * LK + 4 * ty);
      const float2 y2 = *reinterpret_cast<const float2*>(Yt + e * LQ + 2 * tx);
      const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        dp[r][0] = fmaf(vv[r], y2.x, dp[r][0]);
        dp[r][1] = fmaf(vv[r], y2.y, dp[r][1]);
      }
    }
    // p, dS (masked; dropout replays the keep mask of rows q0 + 2tx + u).
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int ql = 2 * tx + u, gi = q0 + ql;
      uint32_t keep = 0xFFu;
      if (p.drop_t != 0 && gi < n)
        keep = keep_byte(p.drop_t, p.seed_lo, p.seed_hi, bh, gi, (j0 + 4 * ty) >> 3);
      const int kshift = (4 * ty) & 7;  // the 4 keys sit in one 8-key group
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int j = j0 + 4 * ty + r;
        float pv = 0.f, ds = 0.f;
        if (gi < n && j < nk && mask.allowed(gi, j)) {
          pv = exp2f(s[r][u] * sl2 - Lv[ql]);
          float dpv = dp[r][u];
          if (p.drop_t != 0) {
            const float xs = ((keep >> (kshift + r)) & 1u) ? p.drop_scale : 0.f;
            dpv *= xs;
            ds = pv * (dpv - Dv[ql]);
            pv *= xs;
          } else {
            ds = pv * (dpv - Dv[ql]);
          }
        }
        Pt[ql * LK + 4 * ty + r] = pv;
        St[ql * LK + 4 * ty + r] = ds;
        Ss[(4 * ty + r) * LQ + ql] = ds;
      }
    }
    __syncthreads();

    // dV += (p xi s)^T dY, dK += dS^T Q over the 32 queries of the tile.
#pragma unroll 4
    for (int q = 0; q < kBQ; ++q) {
      const float4 p4 = *reinterpret_cast<const float4*>(Pt + q * LK + 4 * ty);
      const float4 g4 = *reinterpret_cast<const float4*>(St + q * LK + 4 * ty);
      const float pp[4] = {p4.x, p4.y, p4.z, p4.w};
      const float gg[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
      for (int h = 0; h < CV; ++h) {
        const float4 y4 = *reinterpret_cast<const float4*>(Ys + q * (V + 4) + 64 * h + 4 * tx);
        const float yy[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int e = 0; e < 4; ++e) dv[r][4 * h + e] = fmaf(pp[r], yy[e], dv[r][4 * h + e]);
      }
#pragma unroll
      for (int h = 0; h < CD; ++h) {
        const float4 x4 = *reinterpret_cast<const float4*>(Qs + q * (D + 4) + 64 * h + 4 * tx);
        const float xx[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int e = 0; e < 4; ++e) dk[r][4 * h + e] = fmaf(gg[r], xx[e], dk[r][4 * h + e]);
      }
    }

    // dQ rows 2ty, 2ty+1 of the tile (queries 0..31 over ty 0..15) += dS K.
    {
      float acc[2][4 * CD];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int e = 0; e < 4 * CD; ++e) acc[u][e] = 0.f;
#pragma unroll 4
      for (int key = 0; key < kBK; ++key) {
        const float2 d2 = *reinterpret_cast<const float2*>(Ss + key * LQ + 2 * ty);
#pragma unroll
        for (int h = 0; h < CD; ++h) {
          const float4 k4 = *reinterpret_cast<const float4*>(Ks + key * (D + 4) + 64 * h + 4 * tx);
          const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[0][4 * h + e] = fmaf(d2.x, kk[e], acc[0][4 * h + e]);
            acc[1][4 * h + e] = fmaf(d2.y, kk[e], acc[1][4 * h + e]);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int gi = q0 + 2 * ty + u;
        if (gi < n)
#pragma unroll
          for (int h = 0; h < CD; ++h)
            if (64 * h + 4 * tx < dw)  // dw is a multiple of 4: the 4 columns are all in
              red_add_v4(dQh + (size_t)gi * dw + 64 * h + 4 * tx, c * acc[u][4 * h],
                         c * acc[u][4 * h + 1], c * acc[u][4 * h + 2], c * acc[u][4 * h + 3]);
      }
    }
  }

  // dK = c sum dS^T Q, dV: keys 4ty..4ty+3, columns 4tx.. (+64).
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int j = j0 + 4 * ty + r;
    if (j >= nk) continue;
    T* dKr = static_cast<T*>(a.dK) + ((size_t)bh * nk + j) * dw;
    T* dVr = static_cast<T*>(a.dV) + ((size_t)bh * nk + j) * vw;
#pragma unroll
    for (int h = 0; h < CD; ++h)
      if (64 * h + 4 * tx < dw)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          Elem<T>::store(dKr + 64 * h + 4 * tx + e, c * dk[r][4 * h + e]);
#pragma unroll
    for (int h = 0; h < CV; ++h)
      if (64 * h + 4 * tx < vw)
#pragma unroll
        for (int e = 0; e < 4; ++e) Elem<T>::store(dVr + 64 * h + 4 * tx + e, dv[r][4 * h + e]);
  }
}

template <typename T, int D, int V>
cudaError_t rt_launch(const BwdArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(float) * RtLayout<D, V>::FLOATS;
  auto kern = simt_bwd_rt_kernel<T, D, V>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  before_launch(kKernBwd, s);
  kern<<<dim3((a.p.nk + kBK - 1) / kBK, a.p.BH), kThreads, smem, s>>>(a);
  after_launch(kKernBwd, s);
  return cudaGetLastError();
}

// Kernel widths: 64 for d (or v) <= 64, 128 above.
template <typename T>
cudaError_t rt_dispatch(const BwdArgs& a, cudaStream_t s) {
  const bool d64 = a.p.d <= 64, v64 = a.p.v <= 64;
  if (!d64 && !v64) return rt_launch<T, 128, 128>(a, s);
  if (d64 && v64) return rt_launch<T, 64, 64>(a, s);
  if (!d64) return rt_launch<T, 128, 64>(a, s);
  return rt_launch<T, 64, 128>(a, s);
}

}  // namespace

bool simt_bwd_rt_supported(const Problem& p) {
  return p.d >= 4 && p.v >= 4 && p.d <= 128 && p.v <= 128 && p.d % 4 == 0 && p.v % 4 == 0;
}

cudaError_t launch_simt_bwd_rt(const BwdArgs& a, cudaStream_t s) {
  return a.p.dtype == kF32 ? rt_dispatch<float>(a, s) : rt_dispatch<__nv_bfloat16>(a, s);
}

}  // namespace exattn
