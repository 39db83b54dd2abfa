// Reverse kernel on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// Implements the Reverse procedure of "Exact tiled softmax attention with
// block-recomputed vector-Jacobian products": with the row statistics frozen,
// for every key block J_t and query i it recomputes s_ij from Q and K,
//   p_ij = exp(s_ij - L_i),  gamma_ij = p_ij (G_i . V_j - delta_i),
//   dQ_i += c gamma_ij K_j,  dK_j += c gamma_ij Q_i,  dV_j += p_ij G_i,
// with delta_i = G_i . Y_i precomputed (HarshvardhanJ/FlashAttention,
// backward section).  No n x n matrix exists: one 128 x 128 block at a time.
//
// One CTA = one 128-key block of one (batch, head); it loops over the 128-row
// query blocks that can allow one of its keys.  Per query block i:
//   dP^T = V dY_i^T  -> TMEM B        S^T = K Q_i^T -> TMEM A
//   P^T = exp2(S^T c log2e - L_i log2e), dS^T = P^T o (dP^T - delta_i)
//       (elementwise warps; P^T -> TMEM A, dS^T -> TMEM B and shared memory)
//   dV += P^T dY_i,  dK += dS^T Q_i   (TMEM accumulators for the whole loop)
//   dQ_i = dS K      -> TMEM A, drained by fp32 vector reductions into the
//                       dQ accumulator (scaled by c)
// Warp roles (16 warps; warp w runs on sub-partition w % 4 and reaches TMEM
// lanes 32 (w % 4) ...):
//   warps 0-7   elementwise: thread = key row, warps 0-3 queries 0-63,
//               warps 4-7 queries 64-127; then dV (0-3) / dK (4-7) epilogue
//   warps 8-11  dQ drain: thread = query row
//   warp 12     TMA: K, V once; Q_i, dY_i, delta_i, L_i log2e per block (2 stages)
//   warp 13     MMA issue
// TMEM columns: A [0,128) S^T / P^T / dQ, B [128,256) dP^T / dS^T,
//               dV [256, 256+V), dK [256+V, 256+V+D).
// Every mbarrier wait is bounded (1 s), as in the forward kernel.
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace exattn {

bool make_tmap_bf16(CUtensorMap* m, const void* base, int width, int n, int BH);
bool tmap_encoder_available();

namespace {

using namespace tc;

constexpr int kBM = 128;  // query rows per block
constexpr int kBN = 128;  // keys per CTA
constexpr int kThreads = 512;
constexpr int kWarpTMA = 12;
constexpr int kWarpMMA = 13;
constexpr int kMaxQB = 256;  // query blocks covered by the in-kernel bitmask tile table
constexpr uint32_t kTmemCols = 512;

enum : int { kEmpty = 0, kFull = 1, kPartial = 2 };

struct BwdParams {
  CUtensorMap tq, tk, tv, tdy;
  int n, npad, BH, mask_kind, window, words_per_row;
  const uint32_t* bits;
  const float* delta;  // [BH][npad]
  const float* lse2;   // [BH][npad]
  float sl2;           // c log2(e)
  float scale;         // c
  float* dQacc;        // [BH][n][D]
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  unsigned* status;
};

template <int D, int V>
struct BLayout {
  static constexpr int KBYTES = kBN * D * 2;
  static constexpr int VBYTES = kBN * V * 2;
  static constexpr int QBYTES = kBM * D * 2;
  static constexpr int YBYTES = kBM * V * 2;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KBYTES;
  static constexpr int DS_OFF = V_OFF + VBYTES;
  static constexpr int DSBYTES = kBN * kBM * 2;
  static constexpr int STAGE_OFF = DS_OFF + DSBYTES;
  static constexpr int STAGE = QBYTES + YBYTES;
  static constexpr int VEC_OFF = STAGE_OFF + 2 * STAGE;  // per stage: delta[128], lse2[128]
  static constexpr int BAR_OFF = VEC_OFF + 2 * 1024;
  static constexpr int B_KV = 0, B_QF = 1, B_QE = 3, B_SDP = 5, B_DS = 6, B_DQF = 7, B_DQD = 8,
                       B_DONE = 9, B_DRAIN = 10, NBAR = 11;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;   // [0] tmem base, [1] abort flag
  static constexpr int CLS_OFF = MISC_OFF + 16;         // any bits [8], not-all bits [8]
  static constexpr int TOTAL = CLS_OFF + 2 * (kMaxQB / 32) * 4;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(V == 64 || V == 128, "value dim");
  static_assert(TOTAL <= 232448, "shared memory");
};

__device__ __forceinline__ uint32_t range_bits(int a, int b) {
  a = max(a, 0);
  b = min(b, 31);
  if (a > b) return 0u;
  const uint32_t width = static_cast<uint32_t>(b - a + 1);
  const uint32_t m = width == 32 ? 0xFFFFFFFFu : ((1u << width) - 1u);
  return m << a;
}

// Classification of query block qb against this CTA's key block kb.
__device__ __forceinline__ int classify(const BwdParams& p, int kb, int qb, const uint32_t* anyb,
                                        const uint32_t* notallb) {
  const int n = p.n;
  const int k0 = kb * kBN;
  const bool key_tail = k0 + kBN > n;
  const int k1 = min(k0 + kBN, n) - 1;
  const int q0 = qb * kBM;
  const int q1 = min(q0 + kBM, n) - 1;
  switch (p.mask_kind) {
    case kMaskCausal:
      if (q1 < k0) return kEmpty;
      return (q0 >= k0 + kBN - 1 && !key_tail) ? kFull : kPartial;
    case kMaskWindow:
      if (q1 < k0 || q0 > k1 + p.window - 1) return kEmpty;
      return (q0 >= k0 + kBN - 1 && q1 <= k0 + p.window - 1 && !key_tail) ? kFull : kPartial;
    case kMaskBitmask: {
      if (!((anyb[qb >> 5] >> (qb & 31)) & 1u)) return kEmpty;
      const bool notall = (notallb[qb >> 5] >> (qb & 31)) & 1u;
      return (notall || key_tail) ? kPartial : kFull;
    }
    default:
      return key_tail ? kPartial : kFull;
  }
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int D, int V>
__global__ void __launch_bounds__(kThreads, 1) tc_bwd_kernel(const __grid_constant__ BwdParams p) {
  using Lay = BLayout<D, V>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + Lay::BAR_OFF;
  auto bar = [&](int k) { return bar0 + 8u * k; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  uint32_t* anyb = reinterpret_cast<uint32_t*>(smem + Lay::CLS_OFF);
  uint32_t* notallb = anyb + kMaxQB / 32;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb = blockIdx.x;  // causal: low key blocks have the most query blocks, run first
  const int bh = blockIdx.y;
  const int n = p.n;
  const int k0 = kb * kBN;
  const int nqb = (n + kBM - 1) / kBM;
  int qb_begin = 0, qb_end = nqb;
  if (p.mask_kind == kMaskCausal || p.mask_kind == kMaskWindow) qb_begin = kb;
  if (p.mask_kind == kMaskWindow)
    qb_end = min(nqb, (min(k0 + kBN, n) - 1 + p.window - 1) / kBM + 1);

  if ((sbase & 1023u) != 0u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) raise_status(p.status, kStatusTimeout);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(bar(Lay::B_KV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(Lay::B_QF + s), 1);
      mbar_init(bar(Lay::B_QE + s), 1);
    }
    mbar_init(bar(Lay::B_SDP), 1);
    mbar_init(bar(Lay::B_DS), 8 * 32);
    mbar_init(bar(Lay::B_DQF), 1);
    mbar_init(bar(Lay::B_DQD), 4 * 32);
    mbar_init(bar(Lay::B_DONE), 1);
    mbar_init(bar(Lay::B_DRAIN), 1);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(sbase + Lay::MISC_OFF, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  if (threadIdx.x < 2 * (kMaxQB / 32)) anyb[threadIdx.x] = 0u;
  __syncthreads();
  if (p.mask_kind == kMaskBitmask) {
    // Tile table: for every query block, does a row allow a key of this block,
    // and does every row allow all of its existing keys?  (One warp = 32 rows
    // of one query block.)
    for (int i0 = qb_begin * kBM + warp * 32; i0 < qb_end * kBM; i0 += kThreads) {
      const int i = i0 + lane;
      bool any = false, all = true;
      if (i < n) {
        const uint32_t* row = p.bits + static_cast<size_t>(i) * p.words_per_row;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int w = kb * 4 + q;
          const uint32_t valid = range_bits(0, n - 1 - 32 * w);
          const uint32_t word = w < p.words_per_row ? __ldg(row + w) & valid : 0u;
          any |= word != 0u;
          all &= word == valid;
        }
      }
      const int qb = i0 / kBM;
      const bool wany = __any_sync(0xFFFFFFFFu, any);
      const bool wnotall = __any_sync(0xFFFFFFFFu, i < n && !all);
      if (lane == 0 && wany) atomicOr(&anyb[qb >> 5], 1u << (qb & 31));
      if (lane == 0 && wnotall) atomicOr(&notallb[qb >> 5], 1u << (qb & 31));
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const uint32_t tA = tmem, tB = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + V;

  if (warp == kWarpTMA) {
    if (lane == 0) {
      prefetch_tmap(&p.tq);
      prefetch_tmap(&p.tk);
      prefetch_tmap(&p.tv);
      prefetch_tmap(&p.tdy);
      const uint64_t keep = policy_evict_last();
      mbar_arrive_expect_tx(bar(Lay::B_KV), Lay::KBYTES + Lay::VBYTES);
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(sbase + Lay::K_OFF + c * 16384, &p.tk, bar(Lay::B_KV), 64 * c, k0, bh, keep);
      for (int c = 0; c < V / 64; ++c)
        tma_load_3d(sbase + Lay::V_OFF + c * 16384, &p.tv, bar(Lay::B_KV), 64 * c, k0, bh, keep);
      int it = 0;
      int last_phase[2] = {-1, -1};
      bool ok = true;
      for (int qb = qb_begin; qb < qb_end; ++qb) {
        if (classify(p, kb, qb, anyb, notallb) == kEmpty) continue;
        const int slot = it & 1, phase = (it >> 1) & 1;
        ++it;
        if (!(ok = mbar_wait(bar(Lay::B_QE + slot), phase ^ 1, abort_flag))) break;
        const uint32_t st = sbase + Lay::STAGE_OFF + slot * Lay::STAGE;
        const uint32_t fb = bar(Lay::B_QF + slot);
        mbar_arrive_expect_tx(fb, Lay::QBYTES + Lay::YBYTES + 1024);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(st + c * 16384, &p.tq, fb, 64 * c, qb * kBM, bh, keep);
        for (int c = 0; c < V / 64; ++c)
          tma_load_3d(st + Lay::QBYTES + c * 16384, &p.tdy, fb, 64 * c, qb * kBM, bh, keep);
        const size_t vo = static_cast<size_t>(bh) * p.npad + qb * kBM;
        const uint32_t vec = sbase + Lay::VEC_OFF + slot * 1024;
        bulk_load(vec, p.delta + vo, 512, fb);
        bulk_load(vec + 512, p.lse2 + vo, 512, fb);
        last_phase[slot] = phase;
      }
      if (!ok) {
        raise_status(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      for (int s = 0; s < 2; ++s)
        if (last_phase[s] >= 0) mbar_wait_inflight(bar(Lay::B_QF + s), last_phase[s]);
      mbar_wait(bar(Lay::B_KV), 0, abort_flag);
    }
  } else if (warp == kWarpMMA) {
    if (lane == 0) {
      constexpr uint32_t kIdSS = idesc_bf16(kBN, kBM, false, false);
      constexpr uint32_t kIdDV = idesc_bf16(kBN, V, false, true);
      constexpr uint32_t kIdDK = idesc_bf16(kBN, D, false, true);
      constexpr uint32_t kIdDQ = idesc_bf16(kBM, D, true, true);
      bool ok = mbar_wait(bar(Lay::B_KV), 0, abort_flag);
      tc_fence_after();
      int it = 0;
      for (int qb = qb_begin; qb < qb_end && ok; ++qb) {
        if (classify(p, kb, qb, anyb, notallb) == kEmpty) continue;
        const int slot = it & 1, phase = (it >> 1) & 1;
        const uint32_t st = sbase + Lay::STAGE_OFF + slot * Lay::STAGE;
        if (!(ok = mbar_wait(bar(Lay::B_QF + slot), phase, abort_flag))) break;
        tc_fence_after();
        // dP^T = V dY_i^T (K = v)
#pragma unroll
        for (int kk = 0; kk < V / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tB, sdesc_sw128(sbase + Lay::V_OFF + off, 16, 1024),
                 sdesc_sw128(st + Lay::QBYTES + off, 16, 1024), kIdSS, kk > 0 ? 1u : 0u);
        }
        if (it > 0) {
          if (!(ok = mbar_wait(bar(Lay::B_DQD), (it - 1) & 1, abort_flag))) break;
          tc_fence_after();
        }
        // S^T = K Q_i^T (K = d)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tA, sdesc_sw128(sbase + Lay::K_OFF + off, 16, 1024), sdesc_sw128(st + off, 16, 1024),
                 kIdSS, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(Lay::B_SDP));
        if (!(ok = mbar_wait(bar(Lay::B_DS), it & 1, abort_flag))) break;
        tc_fence_after();
        // dV += P^T dY_i, dK += dS^T Q_i (K = queries, P^T / dS^T from TMEM)
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk) {
          const uint32_t acol = (kk >> 2) * 64 + (kk & 3) * 8;
          mma_ts(tdV, tA + acol, sdesc_sw128(st + Lay::QBYTES + kk * 2048, 16384, 1024), kIdDV,
                 (it > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk) {
          const uint32_t acol = (kk >> 2) * 64 + (kk & 3) * 8;
          mma_ts(tdK, tB + acol, sdesc_sw128(st + kk * 2048, 16384, 1024), kIdDK,
                 (it > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(Lay::B_QE + slot));
        // dQ_i = dS K (K = keys; dS from shared memory, M = queries)
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ss(tA, sdesc_sw128(sbase + Lay::DS_OFF + kk * 2048, 16384, 1024),
                 sdesc_sw128(sbase + Lay::K_OFF + kk * 2048, 16384, 1024), kIdDQ,
                 kk > 0 ? 1u : 0u);
        tc_commit(bar(Lay::B_DQF));
        ++it;
      }
      tc_commit(bar(Lay::B_DONE));
      if (!ok) {
        raise_status(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      tc_commit(bar(Lay::B_DRAIN));
      mbar_wait_inflight(bar(Lay::B_DRAIN), 0);
    }
  } else if (warp < 8) {
    // Elementwise: thread = key row r, query half X.
    const int X = warp >> 2, wl = warp & 3;
    const int r = wl * 32 + lane;
    const int j = k0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(wl * 32) << 16;
    const float sl2 = p.sl2;
    int it = 0;
    bool ok = true;
    for (int qb = qb_begin; qb < qb_end; ++qb) {
      const int cls = classify(p, kb, qb, anyb, notallb);
      if (cls == kEmpty) continue;
      const int slot = it & 1;
      if (!(ok = mbar_wait(bar(Lay::B_SDP), it & 1, abort_flag))) break;
      tc_fence_after();
      const float* dvec = reinterpret_cast<const float*>(smem + Lay::VEC_OFF + slot * 1024);
      const float* lvec = dvec + 128;
      const int q0 = qb * kBM;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int cb = 64 * X + 32 * h;  // first query column of this chunk
        uint32_t s[32], dp[32];
        tmem_ld32(tA + lane_off + cb, s);
        tmem_ld32(tB + lane_off + cb, dp);
        tmem_ld_wait();
        reg_fence(s);
        reg_fence(dp);
        uint32_t allow = 0xFFFFFFFFu;
        if (cls == kPartial) {
          if (j >= n) {
            allow = 0u;
          } else if (p.mask_kind == kMaskCausal) {
            allow = range_bits(j - q0 - cb, 31);
          } else if (p.mask_kind == kMaskWindow) {
            allow = range_bits(j - q0 - cb, j + p.window - 1 - q0 - cb);
          } else if (p.mask_kind == kMaskBitmask) {
            allow = 0u;
            const uint32_t* col = p.bits + (j >> 5);
#pragma unroll 4
            for (int e = 0; e < 32; ++e) {
              const int i = q0 + cb + e;
              if (i < n)
                allow |= ((__ldg(col + static_cast<size_t>(i) * p.words_per_row) >> (j & 31)) & 1u)
                         << e;
            }
          }
        }
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float4 l4 = *reinterpret_cast<const float4*>(lvec + cb + (e & ~3));
          const float4 d4 = *reinterpret_cast<const float4*>(dvec + cb + (e & ~3));
          const float la = (e & 2) ? l4.z : l4.x, lb = (e & 2) ? l4.w : l4.y;
          const float da = (e & 2) ? d4.z : d4.x, db = (e & 2) ? d4.w : d4.y;
          float p0 = ex2(fmaf(__uint_as_float(s[e]), sl2, -la));
          float p1 = ex2(fmaf(__uint_as_float(s[e + 1]), sl2, -lb));
          if (!((allow >> e) & 1u)) p0 = 0.f;
          if (!((allow >> (e + 1)) & 1u)) p1 = 0.f;
          const float g0 = p0 * (__uint_as_float(dp[e]) - da);
          const float g1 = p1 * (__uint_as_float(dp[e + 1]) - db);
          pk[e >> 1] = pack_bf16x2(p0, p1);
          dk[e >> 1] = pack_bf16x2(g0, g1);
        }
        tmem_st16(tA + lane_off + 64 * X + 16 * h, pk);
        tmem_st16(tB + lane_off + 64 * X + 16 * h, dk);
        // dS^T row r, queries cb..cb+31 -> shared memory chunk X (128-byte swizzle).
        uint8_t* drow = smem + Lay::DS_OFF + X * 16384 + r * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = (4 * h + u) ^ (r & 7);
          *reinterpret_cast<uint4*>(drow + unit * 16) =
              make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(Lay::B_DS));
      ++it;
    }
    if (!ok) {
      raise_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    // Epilogue: dV rows (warps 0-3) and dK rows (warps 4-7) of this key block.
    bool have = ok && it > 0;
    if (have) {
      have = mbar_wait(bar(Lay::B_DONE), 0, abort_flag);
      tc_fence_after();
    }
    const int W = X == 0 ? V : D;
    const uint32_t tsrc = (X == 0 ? tdV : tdK) + lane_off;
    const float mul = X == 0 ? 1.f : p.scale;
    __nv_bfloat16* dst = (X == 0 ? p.dV : p.dK) + (static_cast<size_t>(bh) * n + (j < n ? j : 0)) * W;
    for (int ch = 0; ch < W / 32; ++ch) {
      uint32_t o[32];
      if (have) {
        tmem_ld32(tsrc + ch * 32, o);
        tmem_ld_wait();
        reg_fence(o);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
      if (j < n) {
        uint32_t ov[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          ov[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * mul, __uint_as_float(o[2 * e + 1]) * mul);
        uint4* d4 = reinterpret_cast<uint4*>(dst + ch * 32);
#pragma unroll
        for (int e = 0; e < 4; ++e) d4[e] = make_uint4(ov[4 * e], ov[4 * e + 1], ov[4 * e + 2], ov[4 * e + 3]);
      }
    }
  } else if (warp < 12) {
    // dQ drain: thread = query row of the block; c * dQ_i added into the fp32
    // accumulator with 16-byte vector reductions.
    const int wl = warp & 3;
    const int rq = wl * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wl * 32) << 16;
    const float c = p.scale;
    int it = 0;
    bool ok = true;
    for (int qb = qb_begin; qb < qb_end; ++qb) {
      if (classify(p, kb, qb, anyb, notallb) == kEmpty) continue;
      if (!(ok = mbar_wait(bar(Lay::B_DQF), it & 1, abort_flag))) break;
      tc_fence_after();
      const int i = qb * kBM + rq;
      float* dst = p.dQacc + (static_cast<size_t>(bh) * n + (i < n ? i : 0)) * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        tmem_ld32(tA + lane_off + ch * 32, o);
        tmem_ld_wait();
        reg_fence(o);
        if (ch == D / 32 - 1) {
          tc_fence_before();
          mbar_arrive(bar(Lay::B_DQD));
        }
        if (i < n) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            red_add_v4(dst + ch * 32 + e, c * __uint_as_float(o[e]), c * __uint_as_float(o[e + 1]),
                       c * __uint_as_float(o[e + 2]), c * __uint_as_float(o[e + 3]));
        }
      }
      ++it;
    }
    if (!ok) {
      raise_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_d(const BwdArgs& a, cudaStream_t s) {
  const Problem& pr = a.p;
  BwdParams p;
  if (!make_tmap_bf16(&p.tq, a.Q, D, pr.n, pr.BH) || !make_tmap_bf16(&p.tk, a.K, D, pr.n, pr.BH) ||
      !make_tmap_bf16(&p.tv, a.V, D, pr.n, pr.BH) ||
      !make_tmap_bf16(&p.tdy, a.dY, D, pr.n, pr.BH))
    return cudaErrorInvalidValue;
  p.n = pr.n;
  p.npad = a.npad;
  p.BH = pr.BH;
  p.mask_kind = pr.mask_kind;
  p.window = pr.window;
  p.words_per_row = pr.words_per_row;
  p.bits = pr.bitmask;
  p.delta = a.delta;
  p.lse2 = a.lse2;
  p.sl2 = pr.scale * kLog2e;
  p.scale = pr.scale;
  p.dQacc = a.dQacc;
  p.dK = static_cast<__nv_bfloat16*>(a.dK);
  p.dV = static_cast<__nv_bfloat16*>(a.dV);
  p.status = a.status;
  using Lay = BLayout<D, D>;
  auto kern = tc_bwd_kernel<D, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::TOTAL);
  if (e != cudaSuccess) {
    record_error("tc_bwd: cudaFuncSetAttribute", static_cast<int>(e), cudaGetErrorString(e));
    return e;
  }
  dim3 grid((pr.n + kBN - 1) / kBN, pr.BH);
  before_launch(kKernBwd, s);
  kern<<<grid, kThreads, Lay::TOTAL, s>>>(p);
  after_launch(kKernBwd, s);
  return cudaGetLastError();
}

}  // namespace

bool tc_bwd_supported(const Problem& p) {
  if (p.drop_t != 0) return false;  // dropout: SIMT kernels
  if (p.nk != p.n) return false;    // nq != nk: SIMT kernels
  if (p.dtype != kBF16 || p.d != p.v || (p.d != 64 && p.d != 128)) return false;
  if (p.mask_kind == kMaskBitmask && p.n > kMaxQB * kBM) return false;
  return tmap_encoder_available();
}

cudaError_t launch_tc_bwd(const BwdArgs& a, cudaStream_t s) {
  return a.p.d == 128 ? launch_d<128>(a, s) : launch_d<64>(a, s);
}

}  // namespace exattn
