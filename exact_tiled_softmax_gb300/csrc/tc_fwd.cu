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
// Persistent: one CTA per SM takes items from a counter; an item is two
// 128-row query tiles (A, B) of one (batch, head); key blocks of 128.  Each
// tile's output leaves through its own swizzled shared-memory tile and TMA
// stores.  Warp roles (12 warps; warp w runs on sub-partition w % 4):
//   warps 0-3  softmax of tile A (one thread per query row)   warp 8  TMA
//   warps 4-7  softmax of tile B                               warp 9  MMA
// The softmax warpgroups raise their register budget to 208 and the
// producer warpgroup (warps 8-11) lowers its own to 88: each sub-partition
// then holds 2 x 208 x 32 + 88 x 32 = 16128 registers, the 3 x 168 x 32 that
// the CTA was launched with (168 registers a thread).
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
constexpr int kProducerRegs = 88;
constexpr int kWarpTMA = 8;
constexpr int kWarpMMA = 9;
constexpr int kMaxKT = 256;  // key blocks covered by the in-kernel bitmask tile table
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kTmemCols = 512;

enum : int { kEmpty = 0, kFull = 1, kPartial = 2 };

struct FwdParams {
  CUtensorMap tq, tk, tv;
  CUtensorMap ty;  // Y as a store target (not used in summary mode)
  unsigned* sched;  // item counter (zero at launch)
  int n, BH, n_qblocks, mask_kind, window, words_per_row;
  int tile_rows;  // query rows per item: 2 kBM (tiles A and B), or kBM (tile A only)
  int nk, off;  // keys, and the absolute position of query 0 (nk - n)
  int dw, vw;   // columns of Q, K and of V, Y in memory (<= the kernel's D, V)
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

// kSum: the split-KV summary mode, which writes its rows with plain stores:
// no Y staging tiles, and the room goes to a deeper K/V ring (the mode is
// memory-bound).
template <int D, int V, bool kSum = false>
struct Layout {
  static constexpr int DCH = D / 64;
  static constexpr int VCH = V / 64;
  static constexpr int QTILE = kBM * D * 2;
  static constexpr int KBYTES = kBN * D * 2;
  static constexpr int VBYTES = kBN * V * 2;
  static constexpr int SLOT = KBYTES > VBYTES ? KBYTES : VBYTES;
  static constexpr int NSLOT = kSum ? (D == 128 ? 4 : 8) : (D == 128 ? 3 : 6);
  static constexpr int Q_OFF = 0;
  static constexpr int SLOT_OFF = Q_OFF + 2 * QTILE;
  // Y staging tiles, one per row tile: kBM rows as 64-column boxes (128-byte swizzle).
  static constexpr int YST_OFF = SLOT_OFF + NSLOT * SLOT;
  static constexpr int YST = kSum ? 0 : kBM * V * 2;
  static constexpr int BAR_OFF = YST_OFF + 2 * YST;
  // barriers: q_full, q_free, kv_full[NSLOT], kv_empty[NSLOT], s_full[2], p_full[2],
  // o_done[2], o_read[2], item ring full[2] / empty[2], Y tile free[2] / staged[2], drain
  static constexpr int B_Q = 0, B_QFREE = 1, B_KVF = 2, B_KVE = 2 + NSLOT, B_S = 2 + 2 * NSLOT,
                       B_P = B_S + 2, B_O = B_P + 2, B_OREAD = B_O + 2, B_ITEMF = B_OREAD + 2,
                       B_ITEME = B_ITEMF + 2,
                       B_YF = B_ITEME + 2, B_Y = B_YF + 2, B_DRAIN = B_Y + 2, NBAR = B_DRAIN + 1;
  // [0] tmem base, [1] abort flag, [2..3] item ring
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
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

// Item t of the forward -> (row-tile pair x, slice bh, key chunk z).  Items
// come in groups of kHeadGroup slices, so the CTAs at work at one time share
// the K and V rows of a few slices in L2.  Inside the last group the pairs run
// heaviest first over its slices (x = 0 is the last pair of rows: the most key
// blocks under the causal mask), which balances the end of the launch.  Under
// the causal mask the other groups run slice by slice (heaviest pair first in
// each), so that the items reading one slice's K and V run close together:
// measured on B=2 H=32 n=4096, DRAM reads 308 -> 277 MB and the forward 1.3%
// faster; with the full mask, whose items are all alike, the plain order was
// faster.
constexpr int kHeadGroup = 32;

struct FwdItem {
  int bh, split, q0, kt_begin, kt_end;
  TileRows rows[2];
};

__device__ __forceinline__ FwdItem make_item(const FwdParams& p, int t) {
  FwdItem w;
  w.split = t % p.splits;
  t /= p.splits;
  const int per = kHeadGroup * p.n_qblocks;
  const int grp = t / per;
  const int base = grp * kHeadGroup;
  const int hg = min(kHeadGroup, p.BH - base);
  const int r = t - grp * per;
  int x, sl;
  if (p.mask_kind == kMaskCausal && grp < (p.BH + kHeadGroup - 1) / kHeadGroup - 1) {
    sl = r / p.n_qblocks;  // slice by slice
    x = r - sl * p.n_qblocks;
  } else {
    x = r / hg;  // heaviest pairs first over the group's slices
    sl = r - x * hg;
  }
  w.bh = base + sl;
  w.q0 = (p.n_qblocks - 1 - x) * p.tile_rows;
#pragma unroll
  for (int X = 0; X < 2; ++X) {
    w.rows[X].r0 = w.q0 + X * kBM;
    w.rows[X].r1 = min(w.q0 + X * kBM + kBM, p.n) - 1;
    w.rows[X].valid = w.rows[X].r0 < p.n && X * kBM < p.tile_rows;
  }
  const int nkt = (p.nk + kBN - 1) / kBN;
  w.kt_begin = 0;
  w.kt_end = nkt;
  const int alast = (w.rows[1].valid ? w.rows[1].r1 : w.rows[0].r1) + p.off;
  if (p.mask_kind == kMaskCausal || p.mask_kind == kMaskWindow)
    w.kt_end = alast < 0 ? 0 : min(nkt, alast / kBN + 1);
  if (p.mask_kind == kMaskWindow)
    w.kt_begin = max(0, w.rows[0].r0 + p.off - p.window + 1) / kBN;
  if (p.chunk_kt > 0) {
    w.kt_begin = max(w.kt_begin, w.split * p.chunk_kt);
    w.kt_end = max(w.kt_begin, min(w.kt_end, (w.split + 1) * p.chunk_kt));
  }
  return w;
}

template <int D, int V, bool kDrop, bool kSum>
__global__ void __launch_bounds__(kThreads, 1) tc_fwd_kernel(const __grid_constant__ FwdParams p) {
  using Lay = Layout<D, V, kSum>;
  constexpr int NS = Lay::NSLOT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + Lay::BAR_OFF;
  auto bar = [&](int k) { return bar0 + 8u * k; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* item_ring = reinterpret_cast<volatile int*>(misc + 2);  // two entries
  uint32_t* cls_any = reinterpret_cast<uint32_t*>(smem + Lay::CLS_OFF);
  uint32_t* cls_all = cls_any + 2 * (kMaxKT / 32);  // bits set where NOT every pair is allowed

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.n, nk = p.nk;
  // Persistent: the TMA warp takes items from a counter (CTA c starts with
  // item c, then item gridDim.x + the counter's old value) and hands each to
  // the MMA and softmax warps through a two-entry ring in shared memory (-1
  // ends).  The K/V ring and every barrier phase run on across items.
  const int items = p.n_qblocks * p.BH * p.splits;

  if (threadIdx.x == 0) {
    mbar_init(bar(Lay::B_Q), 1);
    mbar_init(bar(Lay::B_QFREE), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(Lay::B_KVF + s), 1);
      mbar_init(bar(Lay::B_KVE + s), 1);
    }
    for (int X = 0; X < 2; ++X) {
      mbar_init(bar(Lay::B_S + X), 1);
      mbar_init(bar(Lay::B_P + X), kBM);
      mbar_init(bar(Lay::B_O + X), 1);
      mbar_init(bar(Lay::B_OREAD + X), kBM);     // tile X's epilogue has waited for O
      mbar_init(bar(Lay::B_ITEMF + X), 1);
      mbar_init(bar(Lay::B_ITEME + X), 1 + 8);  // MMA warp + softmax warps
      mbar_init(bar(Lay::B_YF + X), 1);          // tile X's staging tile is free
      mbar_init(bar(Lay::B_Y + X), kBM);         // tile X's rows are staged
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
    // Tile table of the CTA's one item (the launcher gives every CTA one item
    // for this mask kind): does any row of tile X allow a key of block kt, and
    // do all rows allow every existing key of it?
    const FwdItem w = make_item(p, blockIdx.x);
    const int X = threadIdx.x / kBM;
    const int i = w.q0 + threadIdx.x;
    if (i < n) {
      const uint32_t* row = p.bits + static_cast<size_t>(i) * p.words_per_row;
      // 32 blocks per table word: the row's bits for them are gathered in
      // registers (loads unrolled, so several are in flight) and merged with
      // one shared-memory atomic each.
      for (int k0 = w.kt_begin & ~31; k0 < w.kt_end; k0 += 32) {
        uint32_t anyw = 0u, notallw = 0u;
        const int k1 = min(w.kt_end, k0 + 32);
#pragma unroll 4
        for (int kt = max(k0, w.kt_begin); kt < k1; ++kt) {
          bool any = false, all = true;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int wd = kt * 4 + q;
            const uint32_t valid = range_bits(0, nk - 1 - 32 * wd);
            const uint32_t word = wd < p.words_per_row ? __ldg(row + wd) & valid : 0u;
            any |= word != 0u;
            all &= word == valid;
          }
          anyw |= (any ? 1u : 0u) << (kt & 31);
          notallw |= (all ? 0u : 1u) << (kt & 31);
        }
        const int wd = X * (kMaxKT / 32) + (k0 >> 5);
        if (anyw) atomicOr(&cls_any[wd], anyw);
        if (notallw) atomicOr(&cls_all[wd], notallw);
      }
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  // Consumers: item nitem from the ring (waits for it, then frees the entry).
  auto take_item = [&](int nitem, int& t) {
    const int e = nitem & 1;
    if (!mbar_wait(bar(Lay::B_ITEMF + e), (nitem >> 1) & 1, abort_flag)) return false;
    t = item_ring[e];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(Lay::B_ITEME + e));
    return true;
  };

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
        if (p.chunk_kt == 0) prefetch_tmap(&p.ty);
      }
      const uint64_t keep = policy_evict_last(), stream = policy_evict_first();
      int it = 0, q_loads = 0;
      bool ok = true;
      int t = blockIdx.x;
      for (int nitem = 0;; ++nitem) {
        const int e = nitem & 1;
        if (nitem >= 2 &&
            !(ok = mbar_wait(bar(Lay::B_ITEME + e), ((nitem >> 1) - 1) & 1, abort_flag)))
          break;
        if (leader) {
          item_ring[e] = t < items ? t : -1;
          mbar_arrive(bar(Lay::B_ITEMF + e));
        }
        if (t >= items) break;
        // Claim the next item now; its value is first needed after this one's first block.
        unsigned claimed = 0u;
        if (lane == 0) claimed = atomicAdd(p.sched, 1u);
        const FwdItem w = make_item(p, t);
        // Q of the item once the previous item's S products no longer read Q.
        if (nitem > 0 && !(ok = mbar_wait(bar(Lay::B_QFREE), (nitem - 1) & 1, abort_flag))) break;
        const int nq = w.rows[1].valid ? 2 : 1;
        if (leader) {
          mbar_arrive_expect_tx(bar(Lay::B_Q), nq * Lay::QTILE);
          for (int X = 0; X < nq; ++X)
            for (int c = 0; c < Lay::DCH; ++c)
              tma_load_3d(sbase + Lay::Q_OFF + X * Lay::QTILE + c * 16384, &p.tq, bar(Lay::B_Q),
                          64 * c, w.q0 + X * kBM, w.bh, stream);
        }
        ++q_loads;
        // The next item's Q goes into L2 after this item's first block, so that
        // its load (issued once this item's S products are done) does not wait on HBM.
        int t_next = -1;
        auto prefetch_next = [&]() {
          t_next = static_cast<int>(
              min(__shfl_sync(0xFFFFFFFFu, claimed, 0) + gridDim.x, static_cast<unsigned>(items)));
          if (t_next < items && leader) {
            const FwdItem wn = make_item(p, t_next);
            for (int X = 0; X < 2; ++X)
              if (wn.rows[X].valid)
                for (int c = 0; c < Lay::DCH; ++c)
                  if (64 * c < p.dw) tma_prefetch_3d(&p.tq, 64 * c, wn.q0 + X * kBM, wn.bh);
          }
        };
        for (int kt = w.kt_begin; kt < w.kt_end && ok; ++kt) {
          const int c0 = classify(p, w.rows[0], 0, kt, cls_any, cls_all);
          const int c1 = classify(p, w.rows[1], 1, kt, cls_any, cls_all);
          if (c0 == kEmpty && c1 == kEmpty) continue;
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            const int slot = it % NS, phase = (it / NS) & 1;
            if (!mbar_wait(bar(Lay::B_KVE + slot), phase ^ 1, abort_flag)) {
              ok = false;
              break;
            }
            ++it;  // fills issued
            const uint32_t dst = sbase + Lay::SLOT_OFF + slot * Lay::SLOT;
            if (leader) {
              if (kv == 0) {
                mbar_arrive_expect_tx(bar(Lay::B_KVF + slot), Lay::KBYTES);
                for (int c = 0; c < Lay::DCH; ++c)
                  tma_load_3d(dst + c * 16384, &p.tk, bar(Lay::B_KVF + slot), 64 * c, kt * kBN,
                              w.bh, keep);
              } else {
                mbar_arrive_expect_tx(bar(Lay::B_KVF + slot), Lay::VBYTES);
                for (int c = 0; c < Lay::VCH; ++c)
                  tma_load_3d(dst + c * 16384, &p.tv, bar(Lay::B_KVF + slot), 64 * c, kt * kBN,
                              w.bh, keep);
              }
            }
          }
          if (ok && t_next < 0) prefetch_next();
        }
        if (!ok) break;
        if (t_next < 0) prefetch_next();
        t = t_next;
      }
      __syncwarp();
      if (!ok && leader) {
        raise_status(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      // Never leave with copies in flight: wait (bounded) for the last fill of
      // every slot (fill i = it - 1 - u went to slot i % NS) and for the last Q.
      for (int u = 0; u < NS && u < it; ++u) {
        const int i = it - 1 - u;
        mbar_wait_inflight(bar(Lay::B_KVF + i % NS), (i / NS) & 1);
      }
      if (q_loads > 0) mbar_wait_inflight(bar(Lay::B_Q), (q_loads - 1) & 1);
    } else if (warp == kWarpMMA) {
      constexpr uint32_t kIdescS = idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16(kBM, V, false, true);
      // Descriptors of the Q tiles and of slot 0; slot s and K-step kk only add
      // constants to the start-address field (units of 16 bytes).
      const uint64_t dq0 = sdesc_sw128(sbase + Lay::Q_OFF, 16, 1024);
      const uint64_t dk0 = sdesc_sw128(sbase + Lay::SLOT_OFF, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sbase + Lay::SLOT_OFF, 16384, 1024);
      bool ok = true;
      int it = 0, cnt[2] = {0, 0};
      bool first_pv[2] = {true, true};
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
      for (int nitem = 0; ok; ++nitem) {
        int t;
        if (!(ok = take_item(nitem, t))) break;
        if (t < 0) break;
        const FwdItem w = make_item(p, t);
        // The item's last block with an S product: Q is free once it completes.
        int kt_last = -1;
        for (int kt = w.kt_end - 1; kt >= w.kt_begin; --kt)
          if (classify(p, w.rows[0], 0, kt, cls_any, cls_all) != kEmpty ||
              classify(p, w.rows[1], 1, kt, cls_any, cls_all) != kEmpty) {
            kt_last = kt;
            break;
          }
        if (!(ok = mbar_wait(bar(Lay::B_Q), nitem & 1, abort_flag))) break;
        tc_fence_after();
        first_pv[0] = first_pv[1] = true;
        bool pend_b = false, have_prev = false;
        int pend_b_phase = 0, pend_vslot = 0;
        if (kt_last < 0) commit(Lay::B_QFREE);
        for (int kt = w.kt_begin; kt < w.kt_end && ok; ++kt) {
          const int c0 = classify(p, w.rows[0], 0, kt, cls_any, cls_all);
          const int c1 = classify(p, w.rows[1], 1, kt, cls_any, cls_all);
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
          if (kt == kt_last) commit(Lay::B_QFREE);  // the last S products read Q
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
        // "O done" stays at most one phase ahead of each tile's epilogue, also
        // through items in which a tile has no blocks.
        for (int X = 0; X < 2 && ok; ++X) {
          if (nitem > 0 && !(ok = mbar_wait(bar(Lay::B_OREAD + X), (nitem - 1) & 1, abort_flag)))
            break;
          commit(Lay::B_O + X);
        }
        __syncwarp();
      }
      __syncwarp();
      if (!ok && leader) {
        raise_status(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      // Drain: every MMA issued by this warp has completed before teardown.
      commit(Lay::B_DRAIN);
      mbar_wait_inflight(bar(Lay::B_DRAIN), 0);
    }
  } else {
    // Softmax warpgroups: thread = one query row of tile X.
    regs_inc<kSoftmaxRegs>();
    const int X = warp >> 2;
    const int wl = warp & 3;
    const int r = wl * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wl * 32) << 16;
    const uint32_t t_s = tmem + lane_off + X * kBN;
    const uint32_t t_o = tmem + lane_off + 2 * kBN + X * V;
    const float sl2 = p.sl2;
    int cnt = 0;
    bool ok = true;
    for (int nitem = 0; ok; ++nitem) {
      int t;
      if (!(ok = take_item(nitem, t))) break;
      if (t < 0) break;
      const FwdItem w = make_item(p, t);
      const TileRows mine = w.rows[X];
      const int bh = w.bh;
      const int i = w.q0 + X * kBM + r;
      float m_ref = -INFINITY, l = 0.f;
      const int cnt0 = cnt;
      if (mine.valid) {
        // Key block kt of class c, whose S is in TMEM: P over S's columns, the
        // running maximum and row sum updated.
        // The bit-row words of row i for key block kt (bitmask kind, PARTIAL
        // blocks).  Loaded before the wait for S, so that the loads are in
        // flight while the tensor pipe forms S.
        auto bit_words = [&](int kt, int c, uint32_t (&bw)[4]) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int wd = kt * 4 + q;
            bw[q] = 0xFFFFFFFFu;
            if (p.mask_kind == kMaskBitmask && c == kPartial)
              bw[q] = (i < n && wd < p.words_per_row)
                          ? __ldg(p.bits + static_cast<size_t>(i) * p.words_per_row + wd)
                          : 0u;
          }
        };
        auto block = [&](int kt, int c, const uint32_t (&bw)[4]) {
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
            for (int q = 0; q < 4; ++q)
              mw[q] = range_bits(lo - (k0 + 32 * q), hi - (k0 + 32 * q)) & bw[q];
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
                const uint32_t wd =
                    (e & 3) == 0 ? rw.x : (e & 3) == 1 ? rw.y : (e & 3) == 2 ? rw.z : rw.w;
                pk[e] = pack_bf16x2((wd & 0xFFFFu) >= p.drop_t ? p0 : 0.f,
                                    wd >= (p.drop_t << 16) ? p1 : 0.f);
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
        };
        if constexpr (kDrop) {
          // With dropout the next block is classified while this block's softmax
          // runs (measured: forward 0.943 -> 0.862 ms on the n = 4096 d = 128
          // causal workload; the same form without dropout was 4% slower).
          auto next_block = [&](int kt, int& cls) {
            for (; kt < w.kt_end; ++kt) {
              cls = classify(p, mine, X, kt, cls_any, cls_all);
              if (cls != kEmpty) break;
            }
            return kt;
          };
          int c = kEmpty;
          int kt = next_block(w.kt_begin, c);
          while (kt < w.kt_end) {
            uint32_t bw[4];
            bit_words(kt, c, bw);
            if (!(ok = mbar_wait(bar(Lay::B_S + X), cnt & 1, abort_flag))) break;
            tc_fence_after();
            int c_next = kEmpty;
            const int kt_next = next_block(kt + 1, c_next);
            block(kt, c, bw);
            kt = kt_next;
            c = c_next;
          }
        } else {
          for (int kt = w.kt_begin; kt < w.kt_end; ++kt) {
            const int c = classify(p, mine, X, kt, cls_any, cls_all);
            if (c == kEmpty) continue;
            uint32_t bw[4];
            bit_words(kt, c, bw);
            if (!(ok = mbar_wait(bar(Lay::B_S + X), cnt & 1, abort_flag))) break;
            tc_fence_after();
            block(kt, c, bw);
          }
        }
      }
      if (!ok) break;
      // Epilogue: Y_i = O_i / l_i (bf16), L_i = ln 2 * (m_ref + log2 l_i).  The
      // MMA warp commits O of both tiles every item.
      if (!(ok = mbar_wait(bar(Lay::B_O + X), nitem & 1, abort_flag))) break;
      tc_fence_after();
      const bool have_o = cnt > cnt0;
      const bool valid = mine.valid && i < n;  // tile B of a one-tile item has no rows
      if constexpr (kSum) {
        // Split-KV summary of this key chunk for row i ("Exact tiled softmax
        // attention ...", Forward procedure: the summary of a block of keys).
        const size_t row = (static_cast<size_t>(bh) * p.splits + w.split) * n + (valid ? i : 0);
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
        tc_fence_before();
        mbar_arrive(bar(Lay::B_OREAD + X));
      } else {
        // Rows leave through the row tile's own shared-memory tile in the TMA
        // layout (64-column boxes, 128-byte swizzle) and TMA stores, which write
        // whole lines and clip rows past n.
        const float inv = l > 0.f ? (kDrop ? p.drop_scale : 1.f) / l : 0.f;
        uint32_t yv[V / 2];
        {
          uint32_t o[V / 32][32];
          if (have_o) {
#pragma unroll
            for (int ch = 0; ch < V / 32; ++ch) tmem_ld32(t_o + ch * 32, o[ch]);
            tmem_ld_wait();
#pragma unroll
            for (int ch = 0; ch < V / 32; ++ch) reg_fence(o[ch]);
          } else {
#pragma unroll
            for (int ch = 0; ch < V / 32; ++ch)
#pragma unroll
              for (int e = 0; e < 32; ++e) o[ch][e] = 0u;
          }
#pragma unroll
          for (int e = 0; e < V / 2; ++e)
            yv[e] = pack_bf16x2(__uint_as_float(o[e >> 4][(2 * e) & 31]) * inv,
                                __uint_as_float(o[e >> 4][(2 * e + 1) & 31]) * inv);
        }
        tc_fence_before();  // O read: the next item's first P.V may overwrite it
        mbar_arrive(bar(Lay::B_OREAD + X));
        if (valid) {
          p.L[static_cast<size_t>(bh) * n + i] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
          if (!(l > 0.f)) raise_status(p.status, kStatusEmptyRow);
        }
        // Thread X * kBM issues tile X's stores; its previous ones have read the
        // staging tile before the rows are written again.
        const bool issuer = threadIdx.x == X * kBM;
        if (issuer) {
          bulk_wait_read_all();
          mbar_arrive(bar(Lay::B_YF + X));
        }
        if (!(ok = mbar_wait(bar(Lay::B_YF + X), nitem & 1, abort_flag))) break;
        const uint32_t tile = sbase + Lay::YST_OFF + X * Lay::YST;
#pragma unroll
        for (int u = 0; u < V / 8; ++u) {
          const uint32_t addr = tile + (u >> 3) * (kBM * 128) + r * 128 + (((u & 7) ^ (r & 7)) << 4);
          st_shared_v4(addr, yv[4 * u], yv[4 * u + 1], yv[4 * u + 2], yv[4 * u + 3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(Lay::B_Y + X));
        if (issuer) {
          if (mbar_wait(bar(Lay::B_Y + X), nitem & 1, abort_flag)) {
            if (mine.valid)
#pragma unroll
              for (int c = 0; c < Lay::VCH; ++c)  // no box that starts past Y's columns
                if (64 * c < p.vw)
                  tma_store_3d(&p.ty, tile + c * (kBM * 128), 64 * c, w.q0 + X * kBM, bh);
            bulk_commit();
          } else {
            ok = false;
          }
        }
        ok = __all_sync(0xFFFFFFFFu, ok);
      }
    }
    if (!ok) {
      raise_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    // The stores' issuers: all of their stores complete before the CTA ends.
    if (threadIdx.x == 0 || threadIdx.x == kBM) bulk_wait_all();
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
// swizzle; columns beyond width and rows beyond n read as zeros, and stores clip them.
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

// Widths up to 128 in steps of 8 run on the kernel of width 64 or 128: the
// tensor maps have the true widths, so TMA loads fill the missing columns of
// Q, K and V with zeros (which change neither S nor P.V) and TMA stores clip
// them from Y.
int padded_width(const Problem& p) { return p.d <= 64 && p.v <= 64 ? 64 : 128; }

bool tc_fwd_supported(const Problem& p) {
  if (p.dtype != kBF16 || p.d < 8 || p.v < 8 || p.d > 128 || p.v > 128 || p.d % 8 != 0 ||
      p.v % 8 != 0)
    return false;
  if (!(p.scale > 0.f)) return false;
  if (p.mask_kind == kMaskBitmask && p.nk > kMaxKT * kBN) return false;
  return encode_fn() != nullptr;
}

template <int D>
cudaError_t launch_tc_fwd_d(const FwdArgs& a, cudaStream_t s, int chunk_kt = 0, int splits = 1,
                            float* pm = nullptr, float* pl = nullptr, float* pz = nullptr) {
  const Problem& pr = a.p;
  FwdParams p;
  if (!make_tmap_bf16(&p.tq, a.Q, pr.d, pr.n, pr.BH) ||
      !make_tmap_bf16(&p.tk, a.K, pr.d, pr.nk, pr.BH) ||
      !make_tmap_bf16(&p.tv, a.V, pr.v, pr.nk, pr.BH))
    return cudaErrorInvalidValue;
  p.n = pr.n;
  p.nk = pr.nk;
  p.off = pr.nk - pr.n;
  p.dw = pr.d;
  p.vw = pr.v;
  p.BH = pr.BH;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // Items are pairs of 128-row tiles; a problem with fewer pairs than SMs runs
  // one tile per item instead, which puts up to twice the SMs to work (the
  // second softmax warpgroup of a CTA then idles).
  p.tile_rows = 2 * kBM;
  p.n_qblocks = (pr.n + 2 * kBM - 1) / (2 * kBM);
  if (chunk_kt == 0 && p.n_qblocks * pr.BH < sms && pr.n > kBM) {
    p.tile_rows = kBM;
    p.n_qblocks = (pr.n + kBM - 1) / kBM;
  }
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
  p.splits = chunk_kt > 0 ? splits : 1;
  p.sched = a.status + kSchedWord;
  if (chunk_kt == 0 && !make_tmap_bf16(&p.ty, a.Y, pr.v, pr.n, pr.BH)) return cudaErrorInvalidValue;
  // The summaries are written with the kernel's width: only d = v = D there.
  if (chunk_kt > 0 && (pr.d != D || pr.v != D)) return cudaErrorInvalidValue;
  p.pm = pm;
  p.pl = pl;
  p.pz = pz;
  const bool sum = chunk_kt > 0;
  if (sum && pr.drop_t != 0) return cudaErrorInvalidValue;  // the summaries take no dropout
  auto kern = sum ? tc_fwd_kernel<D, D, false, true>
                  : pr.drop_t != 0 ? tc_fwd_kernel<D, D, true, false>
                                   : tc_fwd_kernel<D, D, false, false>;
  const int alloc = sum ? Layout<D, D, true>::ALLOC : Layout<D, D, false>::ALLOC;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, alloc);
  if (e != cudaSuccess) {
    record_error("tc_fwd: cudaFuncSetAttribute", static_cast<int>(e), cudaGetErrorString(e));
    return e;
  }
  // Persistent: one CTA per SM, items handed out by a counter.  One item per
  // CTA for the bitmask (the kernel builds the CTA's tile table once) and for
  // the split-KV summaries.
  const int items = p.n_qblocks * pr.BH * p.splits;
  int grid = items;
  if (chunk_kt == 0 && pr.mask_kind != kMaskBitmask) grid = items < sms ? items : sms;
  const int role = chunk_kt > 0 ? kKernSplitPartial : kKernFwd;
  before_launch(role, s);
  kern<<<grid, kThreads, alloc, s>>>(p);
  after_launch(role, s);
  return cudaGetLastError();
}

cudaError_t launch_tc_fwd(const FwdArgs& a, cudaStream_t s) {
  return padded_width(a.p) == 128 ? launch_tc_fwd_d<128>(a, s) : launch_tc_fwd_d<64>(a, s);
}

cudaError_t launch_tc_fwd_chunks(const FwdArgs& a, int chunk_keys, int splits, float* pm,
                                 float* pl, float* pz, cudaStream_t s) {
  const int chunk_kt = chunk_keys / kBN;
  return a.p.d == 128 ? launch_tc_fwd_d<128>(a, s, chunk_kt, splits, pm, pl, pz)
                      : launch_tc_fwd_d<64>(a, s, chunk_kt, splits, pm, pl, pz);
}

}  // namespace exattn
