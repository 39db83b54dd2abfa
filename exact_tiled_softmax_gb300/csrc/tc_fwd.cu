// Forward kernel on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// Implements the Forward procedure of "Exact tiled softmax attention with
// block-recomputed vector-Jacobian products" (summary per key block, merge,
// skip blocks with J_t n A_i empty) as the running-statistics recurrence of
// "txf-modern-flash-attention" (Hints): running max, running denominator,
// unnormalised output rescaled by exp(old - new), one division at the end.
// It retains L_i = m_i + ln l_i ("python-flash-attention-online-softmax-
// block-recompute", The fix, item 1).
//
// One CTA = two 128-row query tiles (A, B) of one (batch, head); key blocks
// of 128.  Warp roles (12 warps; warp w runs on sub-partition w % 4):
//   warps 0-3  softmax of tile A (one thread per query row)   warp 8  TMA
//   warps 4-7  softmax of tile B                               warp 9  MMA
// The softmax warpgroups raise their register budget to 208 and the
// producer warpgroup (warps 8-11) lowers its own to 56: each sub-partition
// then holds 2 x 208 x 32 + 56 x 32 <= 16384 registers.
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A, O_B from 256.  P (bf16)
// overwrites the first 64 columns of S and is the TMEM A operand of P.V.
// The MMA warp issues, per key block t:  S_A(t), PV_B(t-1), S_B(t), PV_A(t),
// so each tile's softmax overlaps two MMAs of the other tile.
//
// The reference point of the exponentials is updated lazily: a row keeps its
// old maximum until the new block maximum exceeds it by more than 2^8 (in the
// exp2 domain), so P <= 256 and O is rescaled only on those rare steps.  The
// output and L use the same reference point, so the result is the exact
// softmax in real arithmetic.
//
// Every mbarrier wait is bounded (1 s); on timeout the kernel records
// EXATTN_TIMEOUT in the status word, drains its own copies and MMAs, frees
// TMEM and returns.
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace exattn {
namespace {

using namespace tc;

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per block
constexpr int kThreads = 384;
constexpr int kSoftmaxRegs = 208;
constexpr int kProducerRegs = 56;
constexpr int kWarpTMA = 8;
constexpr int kWarpMMA = 9;
constexpr int kMaxKT = 256;  // key blocks covered by the in-kernel bitmask tile table
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kTmemCols = 512;

enum : int { kEmpty = 0, kFull = 1, kPartial = 2 };

struct FwdParams {
  CUtensorMap tq, tk, tv;
  int n, BH, n_qblocks, mask_kind, window, words_per_row;
  int nk, off;  // keys, and the absolute position of query 0 (nk - n)
  const uint32_t* bits;
  float sl2;  // scale * log2(e), > 0
  __nv_bfloat16* Y;
  float* L;
  unsigned* status;
  uint32_t drop_t, seed_lo, seed_hi;  // dropout (kernel variant kDrop only)
  float drop_scale;
  // Split-KV summary mode (chunk_kt > 0): CTA z covers key blocks
  // [z * chunk_kt, (z + 1) * chunk_kt) and writes its rows' summaries (m in the
  // exp2 domain, l, z unnormalised) to pm / pl / pz [BH][splits][n] instead of Y, L.
  int chunk_kt, splits;
  float* pm;
  float* pl;
  float* pz;
};

template <int D, int V>
struct Layout {
  static constexpr int DCH = D / 64;
  static constexpr int VCH = V / 64;
  static constexpr int QTILE = kBM * D * 2;
  static constexpr int KBYTES = kBN * D * 2;
  static constexpr int VBYTES = kBN * V * 2;
  static constexpr int SLOT = KBYTES > VBYTES ? KBYTES : VBYTES;
  static constexpr int NSLOT = D == 128 ? 4 : 6;
  static constexpr int Q_OFF = 0;
  static constexpr int SLOT_OFF = Q_OFF + 2 * QTILE;
  static constexpr int BAR_OFF = SLOT_OFF + NSLOT * SLOT;
  // barriers: q_full, kv_full[NSLOT], kv_empty[NSLOT], s_full[2], p_full[2], o_done[2], drain
  static constexpr int B_Q = 0, B_KVF = 1, B_KVE = 1 + NSLOT, B_S = 1 + 2 * NSLOT,
                       B_P = B_S + 2, B_O = B_P + 2, B_DRAIN = B_O + 2, NBAR = B_DRAIN + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;   // [0] tmem base, [1] abort flag
  static constexpr int CLS_OFF = (MISC_OFF + 16 + 15) / 16 * 16;
  // Bitmask tile table as bits: any[2][kMaxKT/32], notall[2][kMaxKT/32].
  static constexpr int TOTAL = CLS_OFF + 2 * 2 * (kMaxKT / 32) * 4;
  static constexpr int ALLOC = TOTAL + 1024;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(V == 64 || V == 128, "value dim");
  static_assert(ALLOC <= 232448, "shared memory");
};

// Bits [a, b] (inclusive, may fall outside [0, 31]) of a 32-bit word.
__device__ __forceinline__ uint32_t range_bits(int a, int b) {
  a = max(a, 0);
  b = min(b, 31);
  if (a > b) return 0u;
  const uint32_t width = static_cast<uint32_t>(b - a + 1);
  const uint32_t m = width == 32 ? 0xFFFFFFFFu : ((1u << width) - 1u);
  return m << a;
}

struct TileRows {
  int r0, r1;   // global rows covered (r1 clipped to n-1)
  bool valid;   // at least one row < n
};

// Classification of key block kt for query tile rows [r0, r1]: EMPTY (skip
// the block: J_t n A_i empty for every row), FULL (no masking needed) or
// PARTIAL (mask element by element).  For the bitmask, `any` and `all` are the
// bit tables built by the kernel (`all` holds the NOT-all bits).
__device__ __forceinline__ int classify(const FwdParams& p, const TileRows& t, int X, int kt,
                                        const uint32_t* any, const uint32_t* all) {
  if (!t.valid) return kEmpty;
  const int k0 = kt * kBN;
  const bool tail = k0 + kBN > p.nk;
  const int k1 = min(k0 + kBN, p.nk) - 1;
  const int a0 = t.r0 + p.off, a1 = t.r1 + p.off;  // absolute positions of the rows
  switch (p.mask_kind) {
    case kMaskCausal:
      if (k0 > a1) return kEmpty;
      return (k0 + kBN - 1 <= a0 && !tail) ? kFull : kPartial;
    case kMaskWindow:
      if (k0 > a1 || k1 <= a0 - p.window) return kEmpty;
      return (k0 + kBN - 1 <= a0 && k0 >= a1 - p.window + 1 && !tail) ? kFull : kPartial;
    case kMaskBitmask: {
      const int w = X * (kMaxKT / 32) + (kt >> 5);
      if (!((any[w] >> (kt & 31)) & 1u)) return kEmpty;
      return (((all[w] >> (kt & 31)) & 1u) || tail) ? kPartial : kFull;
    }
    default:
      return tail ? kPartial : kFull;
  }
}

template <int D, int V, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1) tc_fwd_kernel(const __grid_constant__ FwdParams p) {
  using Lay = Layout<D, V>;
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
  uint32_t* cls_all = cls_any + 2 * (kMaxKT / 32);  // bits set where NOT every pair is allowed

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = p.n_qblocks - 1 - blockIdx.x;  // heaviest (causal) query blocks first
  const int bh = blockIdx.y;
  const int q0 = qb * 2 * kBM;
  const int n = p.n;

  TileRows rows[2];
#pragma unroll
  for (int X = 0; X < 2; ++X) {
    rows[X].r0 = q0 + X * kBM;
    rows[X].r1 = min(q0 + X * kBM + kBM, n) - 1;
    rows[X].valid = rows[X].r0 < n;
  }
  const int nk = p.nk;
  const int nkt = (nk + kBN - 1) / kBN;
  int kt_begin = 0, kt_end = nkt;
  {
    const int alast = (rows[1].valid ? rows[1].r1 : rows[0].r1) + p.off;
    if (p.mask_kind == kMaskCausal || p.mask_kind == kMaskWindow)
      kt_end = alast < 0 ? 0 : min(nkt, alast / kBN + 1);
    if (p.mask_kind == kMaskWindow) kt_begin = max(0, rows[0].r0 + p.off - p.window + 1) / kBN;
  }
  const int split = blockIdx.z;
  if (p.chunk_kt > 0) {
    kt_begin = max(kt_begin, split * p.chunk_kt);
    kt_end = max(kt_begin, min(kt_end, (split + 1) * p.chunk_kt));
  }

  if (threadIdx.x == 0) {
    mbar_init(bar(Lay::B_Q), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(Lay::B_KVF + s), 1);
      mbar_init(bar(Lay::B_KVE + s), 1);
    }
    for (int X = 0; X < 2; ++X) {
      mbar_init(bar(Lay::B_S + X), 1);
      mbar_init(bar(Lay::B_P + X), kBM);
      mbar_init(bar(Lay::B_O + X), 1);
    }
    mbar_init(bar(Lay::B_DRAIN), 1);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(sbase + Lay::MISC_OFF, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  if (threadIdx.x < 4 * (kMaxKT / 32)) cls_any[threadIdx.x] = 0u;  // any and not-all bits
  __syncthreads();
  if (p.mask_kind == kMaskBitmask && threadIdx.x < 2 * kBM) {
    // Tile table: does any row of tile X allow a key of block kt, and do all
    // rows allow every existing key of it?
    const int X = threadIdx.x / kBM;
    const int i = q0 + threadIdx.x;
    if (i < n) {
      const uint32_t* row = p.bits + static_cast<size_t>(i) * p.words_per_row;
      for (int kt = kt_begin; kt < kt_end; ++kt) {
        bool any = false, all = true;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int w = kt * 4 + q;
          const uint32_t valid = range_bits(0, nk - 1 - 32 * w);
          const uint32_t word = w < p.words_per_row ? __ldg(row + w) & valid : 0u;
          any |= word != 0u;
          all &= word == valid;
        }
        const int w = X * (kMaxKT / 32) + (kt >> 5);
        if (any) atomicOr(&cls_any[w], 1u << (kt & 31));
        if (!all) atomicOr(&cls_all[w], 1u << (kt & 31));
      }
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp >= 8) {
    regs_dec<kProducerRegs>();
    // The producer warps run their loops on all 32 lanes (warp-uniform state,
    // descriptors in uniform registers); one elected lane issues.
    const bool leader = elect_one();
    if (warp == kWarpTMA) {
      if (leader) {
        prefetch_tmap(&p.tq);
        prefetch_tmap(&p.tk);
        prefetch_tmap(&p.tv);
      }
      const uint64_t keep = policy_evict_last(), stream = policy_evict_first();
      const int nq = rows[1].valid ? 2 : 1;
      if (leader) {
        mbar_arrive_expect_tx(bar(Lay::B_Q), nq * Lay::QTILE);
        for (int X = 0; X < nq; ++X)
          for (int c = 0; c < Lay::DCH; ++c)
            tma_load_3d(sbase + Lay::Q_OFF + X * Lay::QTILE + c * 16384, &p.tq, bar(Lay::B_Q),
                        64 * c, q0 + X * kBM, bh, stream);
      }
      int it = 0;
      int last_phase[NS];
      for (int s = 0; s < NS; ++s) last_phase[s] = -1;
      bool ok = true;
      for (int kt = kt_begin; kt < kt_end && ok; ++kt) {
        const int c0 = classify(p, rows[0], 0, kt, cls_any, cls_all);
        const int c1 = classify(p, rows[1], 1, kt, cls_any, cls_all);
        if (c0 == kEmpty && c1 == kEmpty) continue;
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          const int slot = it % NS, phase = (it / NS) & 1;
          ++it;
          if (!mbar_wait(bar(Lay::B_KVE + slot), phase ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t dst = sbase + Lay::SLOT_OFF + slot * Lay::SLOT;
          if (leader) {
            if (kv == 0) {
              mbar_arrive_expect_tx(bar(Lay::B_KVF + slot), Lay::KBYTES);
              for (int c = 0; c < Lay::DCH; ++c)
                tma_load_3d(dst + c * 16384, &p.tk, bar(Lay::B_KVF + slot), 64 * c, kt * kBN, bh,
                            keep);
            } else {
              mbar_arrive_expect_tx(bar(Lay::B_KVF + slot), Lay::VBYTES);
              for (int c = 0; c < Lay::VCH; ++c)
                tma_load_3d(dst + c * 16384, &p.tv, bar(Lay::B_KVF + slot), 64 * c, kt * kBN, bh,
                            keep);
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
      // Never leave with copies in flight: wait (bounded) for the last fill of
      // every slot and for Q.
      for (int s = 0; s < NS; ++s)
        if (last_phase[s] >= 0) mbar_wait(bar(Lay::B_KVF + s), last_phase[s], abort_flag);
      mbar_wait(bar(Lay::B_Q), 0, abort_flag);
    } else if (warp == kWarpMMA) {
      constexpr uint32_t kIdescS = idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16(kBM, V, false, true);
      // Descriptors of the Q tiles and of slot 0; slot s and K-step kk only add
      // constants to the start-address field (units of 16 bytes).
      const uint64_t dq0 = sdesc_sw128(sbase + Lay::Q_OFF, 16, 1024);
      const uint64_t dk0 = sdesc_sw128(sbase + Lay::SLOT_OFF, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sbase + Lay::SLOT_OFF, 16384, 1024);
      bool ok = mbar_wait(bar(Lay::B_Q), 0, abort_flag);
      tc_fence_after();
      int it = 0, cnt[2] = {0, 0};
      bool first_pv[2] = {true, true};
      bool pend_b = false, have_prev = false;
      int pend_b_phase = 0, pend_vslot = 0;
      auto issue_s = [&](int X, int kslot) {
        const uint64_t a0 = dq0 + static_cast<uint64_t>(X * (Lay::QTILE >> 4));
        const uint64_t b0 = dk0 + static_cast<uint64_t>(kslot * (Lay::SLOT >> 4));
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
            mma_ss(tmem + X * kBN, a0 + off, b0 + off, kIdescS, kk > 0 ? 1u : 0u);
          }
        }
      };
      auto issue_pv = [&](int X, int vslot) {
        const uint64_t b0 = dv0 + static_cast<uint64_t>(vslot * (Lay::SLOT >> 4));
        const uint32_t acc0 = first_pv[X] ? 0u : 1u;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts(tmem + 2 * kBN + X * V, tmem + X * kBN + kk * 8, b0 + kk * 128, kIdescPV,
                   kk == 0 ? acc0 : 1u);
        }
        first_pv[X] = false;
      };
      auto commit = [&](int b) {
        if (leader) tc_commit(bar(b));
      };
      for (int kt = kt_begin; kt < kt_end && ok; ++kt) {
        const int c0 = classify(p, rows[0], 0, kt, cls_any, cls_all);
        const int c1 = classify(p, rows[1], 1, kt, cls_any, cls_all);
        if (c0 == kEmpty && c1 == kEmpty) continue;
        const int kslot = it % NS, kphase = (it / NS) & 1;
        ++it;
        const int vslot = it % NS, vphase = (it / NS) & 1;
        ++it;
        if (!(ok = mbar_wait(bar(Lay::B_KVF + kslot), kphase, abort_flag))) break;
        tc_fence_after();
        if (c0 != kEmpty) {
          issue_s(0, kslot);
          commit(Lay::B_S + 0);
        }
        if (pend_b) {
          if (!(ok = mbar_wait(bar(Lay::B_P + 1), pend_b_phase, abort_flag))) break;
          tc_fence_after();
          issue_pv(1, pend_vslot);
        }
        if (have_prev) commit(Lay::B_KVE + pend_vslot);
        if (c1 != kEmpty) {
          issue_s(1, kslot);
          commit(Lay::B_S + 1);
        }
        commit(Lay::B_KVE + kslot);
        if (!(ok = mbar_wait(bar(Lay::B_KVF + vslot), vphase, abort_flag))) break;
        tc_fence_after();
        if (c0 != kEmpty) {
          if (!(ok = mbar_wait(bar(Lay::B_P + 0), cnt[0] & 1, abort_flag))) break;
          tc_fence_after();
          issue_pv(0, vslot);
          ++cnt[0];
        }
        pend_b = c1 != kEmpty;
        pend_b_phase = cnt[1] & 1;
        if (pend_b) ++cnt[1];
        pend_vslot = vslot;
        have_prev = true;
      }
      if (ok && pend_b) {
        if ((ok = mbar_wait(bar(Lay::B_P + 1), pend_b_phase, abort_flag))) {
          tc_fence_after();
          issue_pv(1, pend_vslot);
        }
      }
      if (ok && have_prev) commit(Lay::B_KVE + pend_vslot);
      commit(Lay::B_O + 0);
      commit(Lay::B_O + 1);
      __syncwarp();
      if (!ok && leader) {
        raise_status(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      // Drain: every MMA issued by this warp has completed before teardown.
      commit(Lay::B_DRAIN);
      mbar_wait(bar(Lay::B_DRAIN), 0, abort_flag);
    }
  } else {
    // Softmax warpgroups: thread = one query row of tile X.
    regs_inc<kSoftmaxRegs>();
    const int X = warp >> 2;
    const TileRows mine = X ? rows[1] : rows[0];
    const int wl = warp & 3;
    const int r = wl * 32 + lane;
    const int i = q0 + X * kBM + r;
    const uint32_t lane_off = static_cast<uint32_t>(wl * 32) << 16;
    const uint32_t t_s = tmem + lane_off + X * kBN;
    const uint32_t t_o = tmem + lane_off + 2 * kBN + X * V;
    const float sl2 = p.sl2;
    float m_ref = -INFINITY, l = 0.f;
    int cnt = 0;
    bool ok = true;
    if (mine.valid) {
      for (int kt = kt_begin; kt < kt_end; ++kt) {
        const int c = classify(p, mine, X, kt, cls_any, cls_all);
        if (c == kEmpty) continue;
        if (!(ok = mbar_wait(bar(Lay::B_S + X), cnt & 1, abort_flag))) break;
        tc_fence_after();
        uint32_t s[128];
        tmem_ld32(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(s + 0));
        tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(s + 32));
        tmem_ld32(t_s + 64, *reinterpret_cast<uint32_t(*)[32]>(s + 64));
        tmem_ld32(t_s + 96, *reinterpret_cast<uint32_t(*)[32]>(s + 96));
        tmem_ld_wait();
        reg_fence(s);
        if (c == kPartial) {
          // Allowed keys of row i in this block as four 32-bit words.
          const int k0 = kt * kBN;
          int lo = 0, hi = nk - 1;
          const int ia = i + p.off;  // absolute position of row i
          if (p.mask_kind == kMaskCausal || p.mask_kind == kMaskWindow) hi = min(hi, ia);
          if (p.mask_kind == kMaskWindow) lo = max(lo, ia - p.window + 1);
          uint32_t mw[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            mw[q] = range_bits(lo - (k0 + 32 * q), hi - (k0 + 32 * q));
            const int w = kt * 4 + q;
            if (p.mask_kind == kMaskBitmask)
              mw[q] &= (i < n && w < p.words_per_row)
                           ? __ldg(p.bits + static_cast<size_t>(i) * p.words_per_row + w)
                           : 0u;
          }
#pragma unroll
          for (int cc = 0; cc < 128; ++cc)
            if (!((mw[cc >> 5] >> (cc & 31)) & 1u)) s[cc] = __float_as_uint(-INFINITY);
        }
        // Row maximum as 8 independent chains of three-input maxima, then a short tree.
        float mx8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = __uint_as_float(s[k]);
#pragma unroll
        for (int cc = 8; cc + 16 <= 128; cc += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mx8[k] = fmax3(mx8[k], __uint_as_float(s[cc + k]), __uint_as_float(s[cc + 8 + k]));
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(mx8[k], __uint_as_float(s[120 + k]));
        const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]),
                               fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
        const float tmax = mx * sl2;  // -inf stays -inf (sl2 > 0)
        const float m_new = fmaxf(m_ref, tmax);
        const bool need = (m_ref != -INFINITY) && (m_new > m_ref + kRescaleThreshold);
        if (m_ref == -INFINITY) m_ref = m_new;
        if (__any_sync(0xFFFFFFFFu, need)) {
          const float alpha = need ? ex2(m_ref - m_new) : 1.f;
          if (need) m_ref = m_new;
          l *= alpha;
#pragma unroll
          for (int ch = 0; ch < V / 32; ++ch) {
            uint32_t o[32];
            tmem_ld32(t_o + ch * 32, o);
            tmem_ld_wait();
            reg_fence(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(t_o + ch * 32, o);
          }
        }
        const float neg = m_ref == -INFINITY ? 0.f : -m_ref;
        float sum2[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};  // partial sums
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
          uint4 rw;  // dropout: Philox words of keys kt*128 + 64*half + 8*(e/4) ..
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            float x0, x1;  // s * c log2(e) - m for the key pair, one packed FMA
            ffma2(x0, x1, __uint_as_float(s[64 * half + 2 * e]),
                  __uint_as_float(s[64 * half + 2 * e + 1]), sl2, sl2, neg, neg);
            const float p0 = ex2(x0);
            const float p1 = ex2(x1);
            // the row sum is of the undropped p (packed adds into 4 pairs of partials)
            fadd2(sum2[e & 3][0], sum2[e & 3][1], sum2[e & 3][0], sum2[e & 3][1], p0, p1);
            if constexpr (kDrop) {
              // Keys 2e and 2e+1 of this half are the low and high halves of one word.
              if ((e & 3) == 0)
                rw = keep_words(p.seed_lo, p.seed_hi, bh, i, kt * (kBN / 8) + 8 * half + e / 4);
              const uint32_t w = (e & 3) == 0 ? rw.x : (e & 3) == 1 ? rw.y : (e & 3) == 2 ? rw.z : rw.w;
              pk[e] = pack_bf16x2((w & 0xFFFFu) >= p.drop_t ? p0 : 0.f,
                                  w >= (p.drop_t << 16) ? p1 : 0.f);
            } else {
              pk[e] = pack_bf16x2(p0, p1);
            }
          }
          tmem_st32(t_s + 32 * half, pk);
        }
        const float rowsum = ((sum2[0][0] + sum2[0][1]) + (sum2[1][0] + sum2[1][1])) +
                             ((sum2[2][0] + sum2[2][1]) + (sum2[3][0] + sum2[3][1]));
        tmem_st_wait();
        l += rowsum;
        tc_fence_before();
        mbar_arrive(bar(Lay::B_P + X));
        ++cnt;
      }
      if (!ok) {
        raise_status(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      // Epilogue: Y_i = O_i / l_i (bf16), L_i = ln 2 * (m_ref + log2 l_i).
      bool have_o = ok && cnt > 0;
      if (have_o) {
        have_o = mbar_wait(bar(Lay::B_O + X), 0, abort_flag);
        tc_fence_after();
      }
      const bool valid = i < n;
      if (p.chunk_kt > 0) {
        // Split-KV summary of this key chunk for row i ("Exact tiled softmax
        // attention ...", Forward procedure: the summary of a block of keys).
        const size_t row = (static_cast<size_t>(bh) * p.splits + split) * n + (valid ? i : 0);
#pragma unroll
        for (int ch = 0; ch < V / 32; ++ch) {
          uint32_t o[32];
          if (have_o) {
            tmem_ld32(t_o + ch * 32, o);
            tmem_ld_wait();
            reg_fence(o);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;
          }
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(p.pz + row * V + ch * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                   __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
          }
        }
        if (valid) {
          p.pm[row] = l > 0.f ? m_ref : -INFINITY;
          p.pl[row] = l;
        }
      } else {
      const float inv = l > 0.f ? (kDrop ? p.drop_scale : 1.f) / l : 0.f;
      __nv_bfloat16* yrow = p.Y + (static_cast<size_t>(bh) * n + (valid ? i : 0)) * V;
#pragma unroll
      for (int ch = 0; ch < V / 32; ++ch) {
        uint32_t o[32];
        if (have_o) {
          tmem_ld32(t_o + ch * 32, o);
          tmem_ld_wait();
          reg_fence(o);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        uint32_t yv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          yv[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(yrow + ch * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(yv[4 * e], yv[4 * e + 1], yv[4 * e + 2], yv[4 * e + 3]);
        }
      }
      if (valid) {
        p.L[static_cast<size_t>(bh) * n + i] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
        if (!(l > 0.f)) raise_status(p.status, kStatusEmptyRow);
      }
      }  // plain epilogue
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

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

}  // namespace

// 3-D bf16 tensor map over [BH][n][width] with 64 x 128 x 1 boxes and 128-byte
// swizzle; rows beyond n read as zeros.
bool make_tmap_bf16(CUtensorMap* m, const void* base, int width, int n, int BH) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(n),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(width) * 2,
                           static_cast<cuuint64_t>(n) * width * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r =
      enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) record_error("cuTensorMapEncodeTiled", static_cast<int>(r), "");
  return r == CUDA_SUCCESS;
}

bool tmap_encoder_available() { return encode_fn() != nullptr; }
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() { return encode_fn(); }

bool tc_fwd_supported(const Problem& p) {
  if (p.dtype != kBF16 || p.d != p.v || (p.d != 64 && p.d != 128)) return false;
  if (!(p.scale > 0.f)) return false;
  if (p.mask_kind == kMaskBitmask && p.nk > kMaxKT * kBN) return false;
  return encode_fn() != nullptr;
}

template <int D>
cudaError_t launch_tc_fwd_d(const FwdArgs& a, cudaStream_t s, int chunk_kt = 0, int splits = 1,
                            float* pm = nullptr, float* pl = nullptr, float* pz = nullptr) {
  const Problem& pr = a.p;
  FwdParams p;
  if (!make_tmap_bf16(&p.tq, a.Q, D, pr.n, pr.BH) || !make_tmap_bf16(&p.tk, a.K, D, pr.nk, pr.BH) ||
      !make_tmap_bf16(&p.tv, a.V, D, pr.nk, pr.BH))
    return cudaErrorInvalidValue;
  p.n = pr.n;
  p.nk = pr.nk;
  p.off = pr.nk - pr.n;
  p.BH = pr.BH;
  p.n_qblocks = (pr.n + 2 * kBM - 1) / (2 * kBM);
  p.mask_kind = pr.mask_kind;
  p.window = pr.window;
  p.words_per_row = pr.words_per_row;
  p.bits = pr.bitmask;
  p.sl2 = pr.scale * kLog2e;
  p.Y = static_cast<__nv_bfloat16*>(a.Y);
  p.L = a.L;
  p.status = a.status;
  p.drop_t = pr.drop_t;
  p.seed_lo = pr.seed_lo;
  p.seed_hi = pr.seed_hi;
  p.drop_scale = pr.drop_scale;
  p.chunk_kt = chunk_kt;
  p.splits = splits;
  p.pm = pm;
  p.pl = pl;
  p.pz = pz;
  using Lay = Layout<D, D>;
  auto kern = pr.drop_t != 0 ? tc_fwd_kernel<D, D, true> : tc_fwd_kernel<D, D, false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::ALLOC);
  if (e != cudaSuccess) {
    record_error("tc_fwd: cudaFuncSetAttribute", static_cast<int>(e), cudaGetErrorString(e));
    return e;
  }
  dim3 grid(p.n_qblocks, pr.BH, chunk_kt > 0 ? splits : 1);
  const int role = chunk_kt > 0 ? kKernSplitPartial : kKernFwd;
  before_launch(role, s);
  kern<<<grid, kThreads, Lay::ALLOC, s>>>(p);
  after_launch(role, s);
  return cudaGetLastError();
}

cudaError_t launch_tc_fwd(const FwdArgs& a, cudaStream_t s) {
  return a.p.d == 128 ? launch_tc_fwd_d<128>(a, s) : launch_tc_fwd_d<64>(a, s);
}

cudaError_t launch_tc_fwd_chunks(const FwdArgs& a, int chunk_keys, int splits, float* pm,
                                 float* pl, float* pz, cudaStream_t s) {
  const int chunk_kt = chunk_keys / kBN;
  return a.p.d == 128 ? launch_tc_fwd_d<128>(a, s, chunk_kt, splits, pm, pl, pz)
                      : launch_tc_fwd_d<64>(a, s, chunk_kt, splits, pm, pl, pz);
}

}  // namespace exattn
