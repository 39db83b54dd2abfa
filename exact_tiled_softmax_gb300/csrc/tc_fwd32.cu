// Forward kernel for fp32 inputs on the sm_103a tensor cores: 3xTF32.
//
// Same method as tc_fwd.cu (the Forward procedure of "Exact tiled softmax
// attention with block-recomputed vector-Jacobian products" as the running-
// statistics recurrence of "txf-modern-flash-attention", Hints; L_i = m_i +
// ln l_i), for fp32 inputs at close to fp32 accuracy.  Each fp32 operand x is
// split into x_hi = x rounded to tf32 (10 fraction bits) and x_lo = (x - x_hi)
// rounded to tf32, and every product of the method is formed from three tf32
// tensor-core products,
//     a b  ~  a_hi b_lo + a_lo b_hi + a_hi b_hi,
// accumulated in fp32 in TMEM, the two small products first.  The dropped
// a_lo b_lo and the rounding of the lo parts each cost about 2^-22 of |a b|.
//
//   S  = Q_hi K_lo^T + Q_lo K_hi^T + Q_hi K_hi^T         (K-steps over d)
//   O += P_hi V_lo   + P_lo V_hi   + P_hi V_hi           (K-steps over keys)
//
// The tensor core's fp32 accumulator drops low-order bits relative to the
// running sum, so a sum over many key blocks would lose accuracy in
// proportion to their number.  Each key block's P V therefore goes into a
// freshly zeroed accumulator O_t, and the softmax threads add it to the
// running O_m with ordinary fp32 arithmetic (promotion of the partial sums,
// applying the rescale factor in the same pass).
//
// A preparation kernel writes K_hi, K_lo ([BH][nk][d]) and V_hi, V_lo
// transposed ([BH][v][nk padded to 32]) to the workspace, so that every
// shared-memory operand is K-major; each softmax thread splits its own Q row
// into Q_hi (TMEM) and Q_lo (shared memory, 128-byte swizzled K-major tile).
// One CTA = one 128-row query tile of one (batch, head); key blocks of 64.
// Warps 0-3: softmax (one thread per query row), warp 4: TMA, warp 5: MMA.
// TMEM (512 columns): Q_hi [0,D), S / P_hi [D,D+64), P_lo [D+64,D+128),
// O_t [D+128, D+128+V), O_m [D+128+V, D+128+2V).  The lazy rescale and the
// masking follow tc_fwd.cu; queries sit at absolute position i + nk - nq.
//
// Every mbarrier wait is bounded (1 s); on timeout the kernel records
// EXATTN_TIMEOUT in the status word, drains its own copies and MMAs, frees
// TMEM and returns.
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace exattn {

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder();  // tc_fwd.cu
bool make_tmap_f32(CUtensorMap* m, const void* base, int inner, int ld, int rows, int BH,
                   int box_rows);

namespace {

using namespace tc;

constexpr int kBM = 128;  // query rows per CTA
constexpr int kBN = 64;   // keys per block
constexpr int kThreads = 192;
constexpr int kWarpTMA = 4;
constexpr int kWarpMMA = 5;
constexpr int kMaxKT = 512;  // key blocks covered by the in-kernel bitmask tile table
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kTmemCols = 512;

enum : int { kEmpty = 0, kFull = 1, kPartial = 2 };

struct Fwd32Params {
  CUtensorMap tkh, tkl, tvh, tvl;
  const float* Q;
  int n, nk, off, BH, mask_kind, window, words_per_row;
  int dw, vw;  // columns of Q, K and of V, Y in memory (multiples of 4, <= the kernel's D, V)
  const uint32_t* bits;
  float sl2;  // scale * log2(e), > 0
  float* Y;
  float* L;
  unsigned* status;
};

template <int D, int V>
struct Layout32 {
  static constexpr int KHALF = kBN * D * 4;  // one of K_hi / K_lo for a block
  static constexpr int VHALF = V * kBN * 4;  // one of V_hi^T / V_lo^T for a block
  static constexpr int SLOT = 2 * (KHALF > VHALF ? KHALF : VHALF);
  static constexpr int NSLOT = D == 128 ? 2 : 5;
  static constexpr int QLO_OFF = 0;              // Q_lo: D/32 chunks of 128 rows x 128 B
  static constexpr int SLOT_OFF = QLO_OFF + kBM * D * 4;
  static constexpr int BAR_OFF = SLOT_OFF + NSLOT * SLOT;
  // barriers: q_ready, kv_full[NSLOT], kv_empty[NSLOT], s_full, p_full, o_done, drain
  static constexpr int B_Q = 0, B_KVF = 1, B_KVE = 1 + NSLOT, B_S = 1 + 2 * NSLOT,
                       B_P = B_S + 1, B_O = B_P + 1, B_DRAIN = B_O + 1, NBAR = B_DRAIN + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;  // [0] tmem base, [1] abort flag
  static constexpr int CLS_OFF = (MISC_OFF + 16 + 15) / 16 * 16;
  static constexpr int TOTAL = CLS_OFF + 2 * (kMaxKT / 32) * 4;
  static constexpr int ALLOC = TOTAL + 1024;
  static constexpr uint32_t T_QH = 0, T_S = D, T_PL = D + kBN, T_OT = D + 2 * kBN,
                            T_OM = D + 2 * kBN + V;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(V == D, "value dim");
  static_assert(T_OM + V <= kTmemCols, "TMEM columns");
  static_assert(ALLOC <= 232448, "shared memory");
};

__device__ __forceinline__ uint32_t range_bits(int a, int b) {
  a = max(a, 0);
  b = min(b, 31);
  if (a > b) return 0u;
  const uint32_t width = static_cast<uint32_t>(b - a + 1);
  const uint32_t m = width == 32 ? 0xFFFFFFFFu : ((1u << width) - 1u);
  return m << a;
}

// Key block kt against query rows [r0, r1] (absolute positions r + off).
__device__ __forceinline__ int classify32(const Fwd32Params& p, int r0, int r1, int kt,
                                          const uint32_t* any, const uint32_t* notall) {
  const int k0 = kt * kBN;
  const bool tail = k0 + kBN > p.nk;
  const int k1 = min(k0 + kBN, p.nk) - 1;
  const int a0 = r0 + p.off, a1 = r1 + p.off;
  switch (p.mask_kind) {
    case kMaskCausal:
      if (k0 > a1) return kEmpty;
      return (k0 + kBN - 1 <= a0 && !tail) ? kFull : kPartial;
    case kMaskWindow:
      if (k0 > a1 || k1 <= a0 - p.window) return kEmpty;
      return (k0 + kBN - 1 <= a0 && k0 >= a1 - p.window + 1 && !tail) ? kFull : kPartial;
    case kMaskBitmask:
      if (!((any[kt >> 5] >> (kt & 31)) & 1u)) return kEmpty;
      return (((notall[kt >> 5] >> (kt & 31)) & 1u) || tail) ? kPartial : kFull;
    default:
      return tail ? kPartial : kFull;
  }
}

template <int D, int V>
__global__ void __launch_bounds__(kThreads, 1)
    tc_fwd32_kernel(const __grid_constant__ Fwd32Params p) {
  using Lay = Layout32<D, V>;
  constexpr int NS = Lay::NSLOT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + Lay::BAR_OFF;
  auto bar = [&](int k) { return bar0 + 8u * k; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  uint32_t* cls_any = reinterpret_cast<uint32_t*>(smem + Lay::CLS_OFF);
  uint32_t* cls_notall = cls_any + kMaxKT / 32;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (p.n + kBM - 1) / kBM;
  const int qb = nqb - 1 - blockIdx.x;  // heaviest (causal) query blocks first
  const int bh = blockIdx.y;
  const int n = p.n, nk = p.nk;
  const int q0 = qb * kBM;
  const int r1 = min(q0 + kBM, n) - 1;
  const int nkt = (nk + kBN - 1) / kBN;
  int kt_begin = 0, kt_end = nkt;
  if (p.mask_kind == kMaskCausal || p.mask_kind == kMaskWindow)
    kt_end = r1 + p.off < 0 ? 0 : min(nkt, (r1 + p.off) / kBN + 1);
  if (p.mask_kind == kMaskWindow)
    kt_begin = min(kt_end, max(0, q0 + p.off - p.window + 1) / kBN);

  if (threadIdx.x == 0) {
    mbar_init(bar(Lay::B_Q), kBM);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(Lay::B_KVF + s), 1);
      mbar_init(bar(Lay::B_KVE + s), 1);
    }
    mbar_init(bar(Lay::B_S), 1);
    mbar_init(bar(Lay::B_P), kBM);
    mbar_init(bar(Lay::B_O), 1);
    mbar_init(bar(Lay::B_DRAIN), 1);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(sbase + Lay::MISC_OFF, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  if (threadIdx.x < 2 * (kMaxKT / 32)) cls_any[threadIdx.x] = 0u;  // any and not-all bits
  __syncthreads();
  if (p.mask_kind == kMaskBitmask && threadIdx.x < kBM) {
    // Tile table: does any row allow a key of block kt, and do all rows allow
    // every existing key of it?  (Two bit-row words per block of 64 keys.)
    const int i = q0 + threadIdx.x;
    if (i < n) {
      const uint32_t* row = p.bits + static_cast<size_t>(i) * p.words_per_row;
      // 32 blocks per table word, gathered in registers (several loads in
      // flight) and merged with one shared-memory atomic each.
      for (int k0 = kt_begin & ~31; k0 < kt_end; k0 += 32) {
        uint32_t anyw = 0u, notallw = 0u;
        const int k1 = min(kt_end, k0 + 32);
#pragma unroll 4
        for (int kt = max(k0, kt_begin); kt < k1; ++kt) {
          bool any = false, all = true;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int w = kt * 2 + q;
            const uint32_t valid = range_bits(0, nk - 1 - 32 * w);
            const uint32_t word = w < p.words_per_row ? __ldg(row + w) & valid : 0u;
            any |= word != 0u;
            all &= word == valid;
          }
          anyw |= (any ? 1u : 0u) << (kt & 31);
          notallw |= (all ? 0u : 1u) << (kt & 31);
        }
        if (anyw) atomicOr(&cls_any[k0 >> 5], anyw);
        if (notallw) atomicOr(&cls_notall[k0 >> 5], notallw);
      }
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  auto cls_of = [&](int kt) { return classify32(p, q0, r1, kt, cls_any, cls_notall); };

  if (warp == kWarpTMA) {
    const bool leader = elect_one();
    if (leader) {
      prefetch_tmap(&p.tkh);
      prefetch_tmap(&p.tkl);
      prefetch_tmap(&p.tvh);
      prefetch_tmap(&p.tvl);
    }
    const uint64_t keep = policy_evict_last();
    int it = 0;
    int last_phase[NS];
    for (int s = 0; s < NS; ++s) last_phase[s] = -1;
    bool ok = true;
    for (int kt = kt_begin; kt < kt_end && ok; ++kt) {
      if (cls_of(kt) == kEmpty) continue;
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        const int slot = it % NS, phase = (it / NS) & 1;
        ++it;
        if (!mbar_wait(bar(Lay::B_KVE + slot), phase ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t dst = sbase + Lay::SLOT_OFF + slot * Lay::SLOT;
        const uint32_t fb = bar(Lay::B_KVF + slot);
        if (leader) {
          if (kv == 0) {  // K_hi, K_lo: D/32 chunks of 64 rows x 128 B each
            mbar_arrive_expect_tx(fb, 2 * Lay::KHALF);
            for (int c = 0; c < D / 32; ++c) {
              tma_load_3d(dst + c * (kBN * 128), &p.tkh, fb, 32 * c, kt * kBN, bh, keep);
              tma_load_3d(dst + Lay::KHALF + c * (kBN * 128), &p.tkl, fb, 32 * c, kt * kBN, bh,
                          keep);
            }
          } else {  // V_hi^T, V_lo^T: two chunks of 32 keys x V rows x 128 B
            mbar_arrive_expect_tx(fb, 2 * Lay::VHALF);
            for (int c = 0; c < kBN / 32; ++c) {
              tma_load_3d(dst + c * (V * 128), &p.tvh, fb, kt * kBN + 32 * c, 0, bh, keep);
              tma_load_3d(dst + Lay::VHALF + c * (V * 128), &p.tvl, fb, kt * kBN + 32 * c, 0, bh,
                          keep);
            }
          }
        }
        last_phase[slot] = phase;
      }
    }
    __syncwarp();
    if (!ok && leader) {
      raise_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    for (int s = 0; s < NS; ++s)
      if (last_phase[s] >= 0) mbar_wait_inflight(bar(Lay::B_KVF + s), last_phase[s]);
  } else if (warp == kWarpMMA) {
    const bool leader = elect_one();
    constexpr uint32_t kIdS = idesc_tf32(kBM, kBN);
    constexpr uint32_t kIdPV = idesc_tf32(kBM, V);
    const uint64_t dslot0 = sdesc_sw128(sbase + Lay::SLOT_OFF, 16, 1024);
    auto commit = [&](int b) {
      if (leader) tc_commit(bar(b));
    };
    // S = Q_hi K_lo^T + Q_lo K_hi^T + Q_hi K_hi^T over D / 8 K-steps each (the
    // two small products first, so that they are summed at their own scale).
    const uint64_t dqlo = sdesc_sw128(sbase + Lay::QLO_OFF, 16, 1024);
    auto issue_s = [&](int kslot) {
      const uint64_t kh = dslot0 + static_cast<uint64_t>((kslot * Lay::SLOT) >> 4);
      const uint64_t kl = kh + static_cast<uint64_t>(Lay::KHALF >> 4);
      if (leader) {
#pragma unroll
        for (int part = 0; part < 3; ++part) {
#pragma unroll
          for (int kk = 0; kk < D / 8; ++kk) {
            const uint32_t off = ((kk >> 2) * (kBN * 128) + (kk & 3) * 32) >> 4;
            const uint32_t acc = (part > 0 || kk > 0) ? 1u : 0u;
            if (part == 1) {  // Q_lo (shared memory) K_hi^T
              const uint32_t qoff = ((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4;
              mma_ss_tf32(tmem + Lay::T_S, dqlo + qoff, kh + off, kIdS, acc);
            } else {          // Q_hi (TMEM) K_lo^T, then Q_hi K_hi^T
              mma_ts_tf32(tmem + Lay::T_S, tmem + Lay::T_QH + 8 * kk, (part == 0 ? kl : kh) + off,
                          kIdS, acc);
            }
          }
        }
      }
    };
    // O_t = P_hi V_lo + P_lo V_hi + P_hi V_hi over kBN / 8 K-steps each (O_t
    // starts from zero for every key block).
    auto issue_pv = [&](int vslot) {
      const uint64_t vh = dslot0 + static_cast<uint64_t>((vslot * Lay::SLOT) >> 4);
      const uint64_t vl = vh + static_cast<uint64_t>(Lay::VHALF >> 4);
      if (leader) {
#pragma unroll
        for (int part = 0; part < 3; ++part) {
          const uint32_t a = tmem + (part == 1 ? Lay::T_PL : Lay::T_S);
          const uint64_t b = part == 0 ? vl : vh;
#pragma unroll
          for (int kk = 0; kk < kBN / 8; ++kk) {
            const uint32_t off = ((kk >> 2) * (V * 128) + (kk & 3) * 32) >> 4;
            mma_ts_tf32(tmem + Lay::T_OT, a + 8 * kk, b + off, kIdPV,
                        (part == 0 && kk == 0) ? 0u : 1u);
          }
        }
      }
    };
    bool ok = mbar_wait(bar(Lay::B_Q), 0, abort_flag);
    tc_fence_after();
    int it = 0, cnt = 0;
    for (int kt = kt_begin; kt < kt_end && ok; ++kt) {
      if (cls_of(kt) == kEmpty) continue;
      const int kslot = it % NS, kphase = (it / NS) & 1;
      ++it;
      const int vslot = it % NS, vphase = (it / NS) & 1;
      ++it;
      if (!(ok = mbar_wait(bar(Lay::B_KVF + kslot), kphase, abort_flag))) break;
      tc_fence_after();
      issue_s(kslot);
      commit(Lay::B_S);
      commit(Lay::B_KVE + kslot);
      if (!(ok = mbar_wait(bar(Lay::B_P), cnt & 1, abort_flag))) break;
      ++cnt;
      if (!(ok = mbar_wait(bar(Lay::B_KVF + vslot), vphase, abort_flag))) break;
      tc_fence_after();
      issue_pv(vslot);
      commit(Lay::B_KVE + vslot);
    }
    commit(Lay::B_O);
    __syncwarp();
    if (!ok && leader) {
      raise_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    commit(Lay::B_DRAIN);
    mbar_wait_inflight(bar(Lay::B_DRAIN), 0);
  } else {
    // Softmax warps: thread = query row r of the tile.
    const int r = warp * 32 + lane;
    const int i = q0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = p.sl2;
    // Q row -> Q_hi in TMEM and Q_lo into row r of the swizzled shared-memory
    // tile (16-byte unit u of a 128-byte row sits at unit u ^ (r % 8)); zeros
    // past the last row.
    {
      const float4* qrow = reinterpret_cast<const float4*>(
          p.Q + (static_cast<size_t>(bh) * n + (i < n ? i : 0)) * p.dw);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t hi[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 x = (i < n && 32 * c + 4 * e < p.dw) ? __ldg(qrow + 8 * c + e)
                                                             : make_float4(0.f, 0.f, 0.f, 0.f);
          const float xs[4] = {x.x, x.y, x.z, x.w};
          float lo4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float h = tf32_hi(xs[u]);
            hi[4 * e + u] = __float_as_uint(h);
            lo4[u] = tf32_lo(xs[u], h);
          }
          *reinterpret_cast<float4*>(smem + Lay::QLO_OFF + c * (kBM * 128) + r * 128 +
                                     ((e ^ (r & 7)) << 4)) =
              make_float4(lo4[0], lo4[1], lo4[2], lo4[3]);
        }
        tmem_st32(tmem + lane_off + Lay::T_QH + 32 * c, hi);
      }
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Lay::B_Q));
    }
    float m_ref = -INFINITY, l = 0.f;
    int cnt = 0;
    bool ok = true;
    for (int kt = kt_begin; kt < kt_end; ++kt) {
      const int c = cls_of(kt);
      if (c == kEmpty) continue;
      if (!(ok = mbar_wait(bar(Lay::B_S), cnt & 1, abort_flag))) break;
      tc_fence_after();
      uint32_t s[kBN];
      tmem_ld32(tmem + lane_off + Lay::T_S, *reinterpret_cast<uint32_t(*)[32]>(s));
      tmem_ld32(tmem + lane_off + Lay::T_S + 32, *reinterpret_cast<uint32_t(*)[32]>(s + 32));
      tmem_ld_wait();
      reg_fence(s);
      if (c == kPartial) {
        const int k0 = kt * kBN;
        int lo = 0, hi = nk - 1;
        const int ia = i + p.off;
        if (p.mask_kind == kMaskCausal || p.mask_kind == kMaskWindow) hi = min(hi, ia);
        if (p.mask_kind == kMaskWindow) lo = max(lo, ia - p.window + 1);
        uint32_t mw[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          mw[q] = range_bits(lo - (k0 + 32 * q), hi - (k0 + 32 * q));
          const int w = kt * 2 + q;
          if (p.mask_kind == kMaskBitmask)
            mw[q] &= (i < n && w < p.words_per_row)
                         ? __ldg(p.bits + static_cast<size_t>(i) * p.words_per_row + w)
                         : 0u;
        }
#pragma unroll
        for (int cc = 0; cc < kBN; ++cc)
          if (!((mw[cc >> 5] >> (cc & 31)) & 1u)) s[cc] = __float_as_uint(-INFINITY);
      }
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = __uint_as_float(s[k]);
#pragma unroll
      for (int cc = 8; cc < kBN; ++cc) mx8[cc & 7] = fmaxf(mx8[cc & 7], __uint_as_float(s[cc]));
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m_new = fmaxf(m_ref, mx * sl2);  // -inf stays -inf (sl2 > 0)
      const bool need = (m_ref != -INFINITY) && (m_new > m_ref + kRescaleThreshold);
      if (m_ref == -INFINITY) m_ref = m_new;
      const float alpha = need ? ex2(m_ref - m_new) : 1.f;
      if (need) m_ref = m_new;
      l *= alpha;
      // Promote the previous block's O_t (stable: the S(t) commit follows every
      // earlier MMA): O_m = (O_m + O_t) * alpha, or O_t * alpha for the first.
      if (cnt > 0) {
#pragma unroll
        for (int ch = 0; ch < V / 32; ++ch) {
          uint32_t ot[32], om[32];
          tmem_ld32(tmem + lane_off + Lay::T_OT + ch * 32, ot);
          if (cnt > 1) tmem_ld32(tmem + lane_off + Lay::T_OM + ch * 32, om);
          tmem_ld_wait();
          reg_fence(ot);
          if (cnt > 1) {
            reg_fence(om);
#pragma unroll
            for (int e = 0; e < 32; ++e)
              om[e] = __float_as_uint((__uint_as_float(om[e]) + __uint_as_float(ot[e])) * alpha);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) om[e] = __float_as_uint(__uint_as_float(ot[e]) * alpha);
          }
          tmem_st32(tmem + lane_off + Lay::T_OM + ch * 32, om);
        }
      }
      const float neg = m_ref == -INFINITY ? 0.f : -m_ref;
      float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t ph[32], pl[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float pv = ex2(fmaf(__uint_as_float(s[32 * half + e]), sl2, neg));
          sum4[e & 3] += pv;
          const float h = tf32_hi(pv);
          ph[e] = __float_as_uint(h);
          pl[e] = __float_as_uint(tf32_lo(pv, h));
        }
        tmem_st32(tmem + lane_off + Lay::T_S + 32 * half, ph);
        tmem_st32(tmem + lane_off + Lay::T_PL + 32 * half, pl);
      }
      tmem_st_wait();
      l += (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
      tc_fence_before();
      mbar_arrive(bar(Lay::B_P));
      ++cnt;
    }
    if (!ok) {
      raise_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    bool have_o = ok && cnt > 0;
    if (have_o) {
      have_o = mbar_wait(bar(Lay::B_O), 0, abort_flag);
      tc_fence_after();
    }
    const bool valid = i < n;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float* yrow = p.Y + (static_cast<size_t>(bh) * n + (valid ? i : 0)) * p.vw;
#pragma unroll
    for (int ch = 0; ch < V / 32; ++ch) {
      uint32_t o[32];
      if (have_o) {  // O = O_m + O_t of the last block
        uint32_t om[32];
        tmem_ld32(tmem + lane_off + Lay::T_OT + ch * 32, o);
        if (cnt > 1) tmem_ld32(tmem + lane_off + Lay::T_OM + ch * 32, om);
        tmem_ld_wait();
        reg_fence(o);
        if (cnt > 1) {
          reg_fence(om);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            o[e] = __float_as_uint(__uint_as_float(om[e]) + __uint_as_float(o[e]));
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
      if (valid) {
        float4* dst = reinterpret_cast<float4*>(yrow + ch * 32);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (32 * ch + 4 * e < p.vw)  // no column past Y's width
            dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv,
                                 __uint_as_float(o[4 * e + 1]) * inv,
                                 __uint_as_float(o[4 * e + 2]) * inv,
                                 __uint_as_float(o[4 * e + 3]) * inv);
      }
    }
    if (valid) {
      p.L[static_cast<size_t>(bh) * n + i] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
      if (!(l > 0.f)) raise_status(p.status, kStatusEmptyRow);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc_fence_after();
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Split K into K_hi, K_lo ([BH][nk][d], same layout) and V into V_hi^T, V_lo^T
// ([BH][v][ldt], keys contiguous): one CTA per (32 keys, batch*head).
__global__ void __launch_bounds__(256) split32_kernel(const float* K, const float* V, float* kh,
                                                      float* kl, float* vth, float* vtl, int nk,
                                                      int d, int v, int ldt) {
  __shared__ float tile[32][257];
  const int bh = blockIdx.y, j0 = blockIdx.x * 32;
  const int rows = min(32, nk - j0);
  const size_t kbase = (static_cast<size_t>(bh) * nk + j0) * d;
  for (int idx = threadIdx.x; idx < rows * d; idx += 256) {
    const float x = __ldg(K + kbase + idx);
    const float h = tf32_hi(x);
    kh[kbase + idx] = h;
    kl[kbase + idx] = tf32_lo(x, h);
  }
  const size_t vbase = (static_cast<size_t>(bh) * nk + j0) * v;
  for (int idx = threadIdx.x; idx < rows * v; idx += 256) tile[idx / v][idx % v] = __ldg(V + vbase + idx);
  __syncthreads();
  const size_t tbase = static_cast<size_t>(bh) * v * ldt + j0;
  for (int idx = threadIdx.x; idx < v * 32; idx += 256) {
    const int c = idx >> 5, jj = idx & 31;
    if (jj < rows) {
      const float x = tile[jj][c];
      const float h = tf32_hi(x);
      vth[tbase + static_cast<size_t>(c) * ldt + jj] = h;
      vtl[tbase + static_cast<size_t>(c) * ldt + jj] = tf32_lo(x, h);
    }
  }
}

template <int D>
cudaError_t launch_d(const FwdArgs& a, const Split32& ws, cudaStream_t s) {
  const Problem& pr = a.p;
  Fwd32Params p;
  // The split arrays keep the true widths; the kernel's loads read zeros for
  // the columns of K and the rows of V^T past them.
  if (!make_tmap_f32(&p.tkh, ws.kh, pr.d, pr.d, pr.nk, pr.BH, kBN) ||
      !make_tmap_f32(&p.tkl, ws.kl, pr.d, pr.d, pr.nk, pr.BH, kBN) ||
      !make_tmap_f32(&p.tvh, ws.vth, pr.nk, ws.ldt, pr.v, pr.BH, D) ||
      !make_tmap_f32(&p.tvl, ws.vtl, pr.nk, ws.ldt, pr.v, pr.BH, D))
    return cudaErrorInvalidValue;
  p.Q = static_cast<const float*>(a.Q);
  p.dw = pr.d;
  p.vw = pr.v;
  p.n = pr.n;
  p.nk = pr.nk;
  p.off = pr.nk - pr.n;
  p.BH = pr.BH;
  p.mask_kind = pr.mask_kind;
  p.window = pr.window;
  p.words_per_row = pr.words_per_row;
  p.bits = pr.bitmask;
  p.sl2 = pr.scale * kLog2e;
  p.Y = static_cast<float*>(a.Y);
  p.L = a.L;
  p.status = a.status;
  using Lay = Layout32<D, D>;
  auto kern = tc_fwd32_kernel<D, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::ALLOC);
  if (e != cudaSuccess) {
    record_error("tc_fwd32: cudaFuncSetAttribute", static_cast<int>(e), cudaGetErrorString(e));
    return e;
  }
  before_launch(kKernSplit32, s);
  split32_kernel<<<dim3((pr.nk + 31) / 32, pr.BH), 256, 0, s>>>(
      static_cast<const float*>(a.K), static_cast<const float*>(a.V), ws.kh, ws.kl, ws.vth,
      ws.vtl, pr.nk, pr.d, pr.v, ws.ldt);
  after_launch(kKernSplit32, s);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  before_launch(kKernFwd, s);
  kern<<<dim3((pr.n + kBM - 1) / kBM, pr.BH), kThreads, Lay::ALLOC, s>>>(p);
  after_launch(kKernFwd, s);
  return cudaGetLastError();
}

}  // namespace

// 3-D fp32 tensor map {inner, rows, BH} with row stride `ld` elements, boxes
// of 32 x box_rows x 1 and 128-byte swizzle; elements past the extents read 0.
bool make_tmap_f32(CUtensorMap* m, const void* base, int inner, int ld, int rows, int BH,
                   int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 4,
                           static_cast<cuuint64_t>(ld) * rows * 4};
  cuuint32_t box[3] = {32, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Widths up to 128 in steps of 4 run on the kernel of width 64 or 128 (zero
// padding, as for bf16): Q rows are loaded and Y rows stored with their own
// widths, and the split copies of K and V keep theirs.
bool tc_fwd32_shape(int d, int v) {
  return d >= 4 && v >= 4 && d <= 128 && v <= 128 && d % 4 == 0 && v % 4 == 0;
}

bool tc_fwd32_supported(const Problem& p) {
  if (p.dtype != kF32 || !tc_fwd32_shape(p.d, p.v)) return false;
  if (!(p.scale > 0.f) || p.drop_t != 0) return false;
  if (p.mask_kind == kMaskBitmask && p.nk > kMaxKT * kBN) return false;
  return tmap_encoder() != nullptr;
}

size_t split32_bytes(const Problem& p) {
  const size_t ldt = (static_cast<size_t>(p.nk) + 31) / 32 * 32;
  const size_t kbytes = 4 * static_cast<size_t>(p.BH) * p.nk * p.d;
  const size_t vbytes = 4 * static_cast<size_t>(p.BH) * p.v * ldt;
  return 2 * ((kbytes + 255) / 256 * 256) + 2 * ((vbytes + 255) / 256 * 256);
}

Split32 split32_layout(const Problem& p, void* base) {
  const size_t ldt = (static_cast<size_t>(p.nk) + 31) / 32 * 32;
  const size_t kbytes = (4 * static_cast<size_t>(p.BH) * p.nk * p.d + 255) / 256 * 256;
  const size_t vbytes = (4 * static_cast<size_t>(p.BH) * p.v * ldt + 255) / 256 * 256;
  char* b = static_cast<char*>(base);
  Split32 w;
  w.kh = reinterpret_cast<float*>(b);
  w.kl = reinterpret_cast<float*>(b + kbytes);
  w.vth = reinterpret_cast<float*>(b + 2 * kbytes);
  w.vtl = reinterpret_cast<float*>(b + 2 * kbytes + vbytes);
  w.ldt = static_cast<int>(ldt);
  return w;
}

cudaError_t launch_tc_fwd32(const FwdArgs& a, const Split32& ws, cudaStream_t s) {
  return a.p.d <= 64 && a.p.v <= 64 ? launch_d<64>(a, ws, s) : launch_d<128>(a, ws, s);
}

}  // namespace exattn
