// Reverse pass on the sm_103a tensor cores as two kernels without atomics.
//
// Implements the Reverse procedure of "Exact tiled softmax attention with
// block-recomputed vector-Jacobian products" with frozen statistics:
//   p_ij = exp(s_ij - L_i),  gamma_ij = p_ij (G_i . V_j - delta_i),
//   dK_j += c gamma_ij Q_i,  dV_j += p_ij G_i     (tc_bwd_kv_kernel, key-major)
//   dQ_i += c gamma_ij K_j                         (tc_bwd_q_kernel, query-major)
// with delta_i = G_i . Y_i (HarshvardhanJ/FlashAttention, backward section).
// Each kernel recomputes the probability block it needs; neither stores an
// n x n matrix, and dQ is written once per query block, so no fp32
// accumulator or reductions are needed.  The dQ kernel runs first: it also
// forms delta_i and L_i log2(e) for its query block and writes both for the
// dK/dV kernel.
//
// Both kernels are persistent: one CTA per SM takes items (a block of 128 keys
// or queries of one slice) from a counter in the workspace, in groups of 16
// slices with the heaviest causal blocks first, and hands them to its warps
// through a two-entry ring in shared memory.  Results leave through swizzled
// shared-memory tiles and TMA stores.
// tc_bwd_kv_kernel -- item = a 128-key block; loop over query blocks.
//   TMEM: A [0,128) S^T then P^T (bf16), B [128,256) dP^T then dS^T (bf16),
//   dV [256, 256+V), dK [256+V, 256+V+D).  S^T and dP^T cover the block's 128
//   queries (K and V are read once per block); the issue order
//   S(0) dP(0) | dV(0) S(1) dK(0) dP(1) | ... relies on the in-order tensor
//   pipe, so the MMAs of one block overlap the elementwise work of the next.
// tc_bwd_q_kernel -- item = a 128-query block; loop over key blocks.
//   K and V in separate rings (3 + 1 slots for d = 128): V(t) is read only by
//   dP(t), K(t) until dQ(t).
//   TMEM: S [0,128), dP double buffer [128,256) and [256,384) (dS bf16 is
//   written over its own dP), dQ [384, 384+D).  S(t+1) is issued as soon as
//   the elementwise warps hold S(t) in registers (before they compute dS(t));
//   dP(t+1) goes into the other buffer even earlier.
// Warp roles (both kernels, 18 warps): warps 0-15 elementwise, four groups of
// 32 columns (group = warp / 4, TMEM lane quarter = warp % 4); warp 16 TMA;
// warp 17 MMA.  The producer warps run warp-uniform loops and one elected
// lane issues.  Every mbarrier wait is bounded (1 s).
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace exattn {

bool make_tmap_bf16(CUtensorMap* m, const void* base, int width, int n, int BH);
bool tmap_encoder_available();

namespace {

using namespace tc;

constexpr int kBM = 128;  // queries per block
constexpr int kBN = 128;  // keys per block
constexpr int kThreads = 576;
constexpr int kEwWarps = 16;
constexpr int kWarpTMA = 16;
constexpr int kWarpMMA = 17;
constexpr int kMaxBlocks = 256;  // blocks covered by the in-kernel bitmask tile table
constexpr uint32_t kTmemCols = 512;

enum : int { kEmpty = 0, kFull = 1, kPartial = 2 };

struct Bwd2Params {
  CUtensorMap tq, tk, tv, tdy;
  CUtensorMap tdk, tdv;  // dK, dV as store targets (dK/dV kernel)
  CUtensorMap tdq;       // dQ as a store target (dQ kernel)
  CUtensorMap ty;        // Y, for the dQ kernel's L2 prefetch of the next item's rows
  int n, npad, BH, mask_kind, window, words_per_row;
  int d;  // columns of Q, K, dQ and dK in memory (<= the kernel's D; TMA fills the rest with zeros)
  int v;  // columns of V, Y, dY and dV in memory (<= the kernel's V, likewise)
  int nk, off;  // keys, and the absolute position of query 0 (nk - n)
  const uint32_t* bits;
  float* delta;  // [BH][npad]: written by the dQ kernel, read by the dK/dV kernel
  float* lse2;   // [BH][npad]  L log2(e), +inf on padding / empty rows (same)
  const __nv_bfloat16* Y;  // [BH][n][V], for delta_i = dY_i . Y_i
  const float* L;          // [BH][n], natural log
  float sl2;           // c log2(e)
  float scale;         // c
  __nv_bfloat16* dQ;
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  unsigned* status;
  unsigned* sched;  // item counters of the dK/dV ([0]) and dQ ([1]) kernels (zero at launch)
  uint32_t drop_t, seed_lo, seed_hi;  // dropout (kernel variants kDrop only)
  float drop_scale;
};

// 32 x 32 bit-matrix transpose across a warp: on return bit e of lane L is bit
// L of lane e's input.  Five butterfly steps, each swapping the off-diagonal
// j x j blocks of lane pairs (L, L ^ j).
__device__ __forceinline__ uint32_t transpose_bits32(uint32_t x, int lane) {
  constexpr uint32_t kM[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int k = 0; k < 5; ++k) {
    const int j = 16 >> k;
    const uint32_t m = kM[k];
    const uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, x, j);
    x = (lane & j) ? ((x & ~m) | ((y >> j) & m)) : ((x & m) | ((y & m) << j));
  }
  return x;
}

// Keep bits of keys j0 .. j0+31 (j0 a multiple of 8) of query row i: bit e is key j0 + e.
__device__ __forceinline__ uint32_t keep_word32(const Bwd2Params& p, int bh, int i, int j0) {
  uint32_t w = 0;
#pragma unroll 1
  for (int g = 0; g < 4; ++g)
    w |= keep_byte(p.drop_t, p.seed_lo, p.seed_hi, bh, i, (j0 >> 3) + g) << (8 * g);
  return w;
}

__device__ __forceinline__ uint32_t range_bits(int a, int b) {
  a = max(a, 0);
  b = min(b, 31);
  if (a > b) return 0u;
  const uint32_t width = static_cast<uint32_t>(b - a + 1);
  const uint32_t m = width == 32 ? 0xFFFFFFFFu : ((1u << width) - 1u);
  return m << a;
}

// Classification of the (query block qb, key block kb) tile.  Bitmask tiles
// come from a table the kernel builds (bit t of any/notall for block t of the
// loop dimension).
__device__ __forceinline__ int classify_tile(const Bwd2Params& p, int qb, int kb, bool any_bit,
                                             bool notall_bit) {
  const int k0 = kb * kBN;
  const bool key_tail = k0 + kBN > p.nk;
  const int k1 = min(k0 + kBN, p.nk) - 1;
  const int q0 = qb * kBM + p.off;                  // absolute positions of the
  const int q1 = min(qb * kBM + kBM, p.n) - 1 + p.off;  // block's first and last rows
  switch (p.mask_kind) {
    case kMaskCausal:
      if (q1 < k0) return kEmpty;
      return (q0 >= k0 + kBN - 1 && !key_tail) ? kFull : kPartial;
    case kMaskWindow:
      if (q1 < k0 || q0 > k1 + p.window - 1) return kEmpty;
      return (q0 >= k0 + kBN - 1 && q1 <= k0 + p.window - 1 && !key_tail) ? kFull : kPartial;
    case kMaskBitmask:
      if (!any_bit) return kEmpty;
      return (notall_bit || key_tail) ? kPartial : kFull;
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

// Bitmask tile table for one CTA: for each block t of the loop range, does any
// (query, key) pair of the tile allow attention, and is some existing pair
// not allowed?  key_major: the CTA owns key block `fixed` and loops over query
// blocks; otherwise it owns query block `fixed` and loops over key blocks.
__device__ void build_bitmask_table(const Bwd2Params& p, bool key_major, int fixed, int t_begin,
                                    int t_end, uint32_t* anyb, uint32_t* notallb) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.n;
  if (key_major) {
    // One warp = 32 query rows of one query block; key words of block `fixed`.
    for (int i0 = t_begin * kBM + warp * 32; i0 < t_end * kBM; i0 += kThreads) {
      const int i = i0 + lane;
      bool any = false, all = true;
      if (i < n) {
        const uint32_t* row = p.bits + static_cast<size_t>(i) * p.words_per_row;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int w = fixed * 4 + q;
          const uint32_t valid = range_bits(0, p.nk - 1 - 32 * w);
          const uint32_t word = w < p.words_per_row ? __ldg(row + w) & valid : 0u;
          any |= word != 0u;
          all &= word == valid;
        }
      }
      const int t = i0 / kBM;
      const bool wany = __any_sync(0xFFFFFFFFu, any);
      const bool wnotall = __any_sync(0xFFFFFFFFu, i < n && !all);
      if (lane == 0 && wany) atomicOr(&anyb[t >> 5], 1u << (t & 31));
      if (lane == 0 && wnotall) atomicOr(&notallb[t >> 5], 1u << (t & 31));
    }
  } else {
    // The CTA's 128 query rows; thread = (row, key block) pairs.
    for (int idx = threadIdx.x; idx < kBM * (t_end - t_begin); idx += kThreads) {
      const int r = idx % kBM;
      const int t = t_begin + idx / kBM;
      const int i = fixed * kBM + r;
      if (i >= n) continue;
      const uint32_t* row = p.bits + static_cast<size_t>(i) * p.words_per_row;
      bool any = false, all = true;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int w = t * 4 + q;
        const uint32_t valid = range_bits(0, p.nk - 1 - 32 * w);
        const uint32_t word = w < p.words_per_row ? __ldg(row + w) & valid : 0u;
        any |= word != 0u;
        all &= word == valid;
      }
      if (any) atomicOr(&anyb[t >> 5], 1u << (t & 31));
      if (!all) atomicOr(&notallb[t >> 5], 1u << (t & 31));
    }
  }
}

// =========================================================================
// Key-major kernel: dK, dV
// =========================================================================
template <int D, int V>
struct KvLayout {
  static constexpr int KBYTES = kBN * D * 2;
  static constexpr int VBYTES = kBN * V * 2;
  static constexpr int QBYTES = kBM * D * 2;
  static constexpr int YBYTES = kBM * V * 2;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KBYTES;
  static constexpr int STAGE_OFF = V_OFF + VBYTES;
  static constexpr int STAGE = QBYTES + YBYTES;
  static constexpr int NST = 2;
  static constexpr int VEC_OFF = STAGE_OFF + NST * STAGE;  // per stage: delta[128], lse2[128]
  // Epilogue tile: kBN rows of dV, then of dK, as 64-column boxes (128-byte swizzle).
  static constexpr int EPI_OFF = VEC_OFF + NST * 1024;
  static constexpr int EPI = kBN * (D > V ? D : V) * 2;
  static constexpr int BAR_OFF = EPI_OFF + EPI;
  // B_S, B_DP: S^T(i), dP^T(i) complete (MMA commits); B_P, B_DSB: P^T(i), dS^T(i)
  // written to TMEM (elementwise arrivals).
  static constexpr int B_KV = 0, B_QF = 1, B_QE = B_QF + NST, B_S = B_QE + NST, B_DP = B_S + 1,
                       B_P = B_DP + 1, B_DSB = B_P + 1,
                       B_DONE = B_DSB + 1, B_DRAIN = B_DONE + 1, B_KVFREE = B_DRAIN + 1,
                       B_ACCFREE = B_KVFREE + 1, B_ITEMF = B_ACCFREE + 1, B_ITEME = B_ITEMF + 2,
                       B_EPIFV = B_ITEME + 2, B_EPIV = B_EPIFV + 1, B_EPIFK = B_EPIV + 1,
                       B_EPIK = B_EPIFK + 1, NBAR = B_EPIK + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int CLS_OFF = MISC_OFF + 16;
  static constexpr int TOTAL = CLS_OFF + 2 * (kMaxBlocks / 32) * 4;
  static_assert(TOTAL <= 232448, "shared memory");
};

// Item t of the persistent dK/dV kernel -> (key block kb, slice bh).  Items
// come in groups of kHeadGroup slices; inside a group the key blocks ascend
// (under the causal mask the low ones reach the most query blocks), so the
// CTAs at work at one time share the Q and dY rows of a few slices in L2.
constexpr int kHeadGroup = 16;
__device__ __forceinline__ void kv_item(int t, int nkb, int BH, int& kb, int& bh) {
  const int per = kHeadGroup * nkb;
  const int grp = t / per;
  const int base = grp * kHeadGroup;
  const int hg = min(kHeadGroup, BH - base);
  const int r = t - grp * per;
  kb = r / hg;
  bh = base + (r - kb * hg);
}

template <int D, int V, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_kv_kernel(const __grid_constant__ Bwd2Params p) {
  using Lay = KvLayout<D, V>;
  constexpr int NST = Lay::NST;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + Lay::BAR_OFF;
  auto bar = [&](int k) { return bar0 + 8u * k; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* item_ring = reinterpret_cast<volatile int*>(misc + 2);  // two entries
  uint32_t* anyb = reinterpret_cast<uint32_t*>(smem + Lay::CLS_OFF);
  uint32_t* notallb = anyb + kMaxBlocks / 32;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.n, nk = p.nk, off = p.off;
  const int nqb = (n + kBM - 1) / kBM, nkb = (nk + kBN - 1) / kBN;
  const int items = nkb * p.BH;
  // Persistent: the TMA warp takes items from a counter (CTA c starts with
  // item c, then item gridDim.x + the counter's old value) and hands each
  // to the other roles through a two-entry ring in shared memory (-1 ends).
  // Ring and barrier phases run on across items.
  // Query blocks that can reach key block kb (row i sits at i + off).
  auto q_range = [&](int kb, int& qb_begin, int& qb_end) {
    const int k0 = kb * kBN;
    qb_begin = 0;
    qb_end = nqb;
    if (p.mask_kind == kMaskCausal || p.mask_kind == kMaskWindow)
      qb_begin = min(nqb, max(0, k0 - off) / kBM);
    if (p.mask_kind == kMaskWindow) {
      const int last = min(k0 + kBN, nk) - 1 - off + p.window - 1;
      qb_end = last < 0 ? 0 : min(nqb, last / kBM + 1);
    }
  };

  if ((sbase & 1023u) != 0u) {
    if (threadIdx.x == 0) raise_status(p.status, kStatusTimeout);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(bar(Lay::B_KV), 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar(Lay::B_QF + s), 1);
      mbar_init(bar(Lay::B_QE + s), 1);
    }
    mbar_init(bar(Lay::B_S), 1);
    mbar_init(bar(Lay::B_DP), 1);
    mbar_init(bar(Lay::B_P), kEwWarps * 32);
    mbar_init(bar(Lay::B_DSB), kEwWarps * 32);
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(Lay::B_ITEMF + h), 1);
      mbar_init(bar(Lay::B_ITEME + h), 1 + kEwWarps);  // MMA warp + elementwise warps
    }
    mbar_init(bar(Lay::B_DONE), 1);
    mbar_init(bar(Lay::B_DRAIN), 1);
    mbar_init(bar(Lay::B_KVFREE), 1);
    mbar_init(bar(Lay::B_ACCFREE), kEwWarps * 32);
    mbar_init(bar(Lay::B_EPIFV), 1);   // the dK store of the previous item has read the tile
    mbar_init(bar(Lay::B_EPIV), 8 * 32);
    mbar_init(bar(Lay::B_EPIFK), 1);   // the dV store has read the tile
    mbar_init(bar(Lay::B_EPIK), 8 * 32);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(sbase + Lay::MISC_OFF, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  if (threadIdx.x < 2 * (kMaxBlocks / 32)) anyb[threadIdx.x] = 0u;
  __syncthreads();
  if (p.mask_kind == kMaskBitmask) {
    // The bitmask tile table is per key block: the launcher gives every CTA
    // exactly one item for this mask kind (item blockIdx.x).
    int kb0, bh0, qb_begin, qb_end;
    kv_item(blockIdx.x, nkb, p.BH, kb0, bh0);
    q_range(kb0, qb_begin, qb_end);
    build_bitmask_table(p, true, kb0, qb_begin, qb_end, anyb, notallb);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const uint32_t tA = tmem, tB = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + V;
  auto cls_of = [&](int qb, int kb) {
    return classify_tile(p, qb, kb, (anyb[qb >> 5] >> (qb & 31)) & 1u,
                         (notallb[qb >> 5] >> (qb & 31)) & 1u);
  };
  // Consumers: item nitem from the ring (waits for it, then frees the entry).
  auto take_item = [&](int nitem, int& t) {
    const int e = nitem & 1;
    if (!mbar_wait(bar(Lay::B_ITEMF + e), (nitem >> 1) & 1, abort_flag)) return false;
    t = item_ring[e];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(Lay::B_ITEME + e));
    return true;
  };

  if (warp == kWarpTMA) {
    const bool leader = elect_one();
    if (leader) {
      prefetch_tmap(&p.tq);
      prefetch_tmap(&p.tk);
      prefetch_tmap(&p.tv);
      prefetch_tmap(&p.tdy);
      prefetch_tmap(&p.tdk);
      prefetch_tmap(&p.tdv);
    }
    const uint64_t keep = policy_evict_last();   // Q, dY: read by every key block of the slice
    const uint64_t once = policy_evict_first();  // K, V: read by one item
    int it = 0, kv_loads = 0;
    bool ok = true;
    int t = blockIdx.x;
    for (int nitem = 0;; ++nitem) {
      const int e = nitem & 1;
      if (nitem >= 2 && !(ok = mbar_wait(bar(Lay::B_ITEME + e), ((nitem >> 1) - 1) & 1, abort_flag)))
        break;
      if (leader) {
        item_ring[e] = t < items ? t : -1;
        mbar_arrive(bar(Lay::B_ITEMF + e));
      }
      if (t >= items) break;
      // Claim the next item now; its value is first needed after this one.
      unsigned claimed = 0u;
      if (lane == 0) claimed = atomicAdd(p.sched, 1u);
      int kb, bh;
      kv_item(t, nkb, p.BH, kb, bh);
      const int k0 = kb * kBN;
      int qb_begin, qb_end;
      q_range(kb, qb_begin, qb_end);
      // K and V of the item once the previous item's S^T, dP^T products no longer read them.
      if (nitem > 0 && !(ok = mbar_wait(bar(Lay::B_KVFREE), (nitem - 1) & 1, abort_flag))) break;
      if (leader) {
        mbar_arrive_expect_tx(bar(Lay::B_KV), Lay::KBYTES + Lay::VBYTES);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sbase + Lay::K_OFF + c * 16384, &p.tk, bar(Lay::B_KV), 64 * c, k0, bh, once);
        for (int c = 0; c < V / 64; ++c)
          tma_load_3d(sbase + Lay::V_OFF + c * 16384, &p.tv, bar(Lay::B_KV), 64 * c, k0, bh, once);
      }
      ++kv_loads;
      // The next item's K and V go into L2 after this item's first stage load,
      // so that their load (issued once this item's last S^T, dP^T products are done)
      // does not wait on HBM.
      int t_next = -1;
      auto prefetch_next = [&]() {
        t_next = static_cast<int>(
            min(__shfl_sync(0xFFFFFFFFu, claimed, 0) + gridDim.x, static_cast<unsigned>(items)));
        if (t_next < items && leader) {
          int kbn, bhn;
          kv_item(t_next, nkb, p.BH, kbn, bhn);
          for (int c = 0; c < D / 64; ++c)
            if (64 * c < p.d) tma_prefetch_3d(&p.tk, 64 * c, kbn * kBN, bhn);
          for (int c = 0; c < V / 64; ++c)
            if (64 * c < p.v) tma_prefetch_3d(&p.tv, 64 * c, kbn * kBN, bhn);
        }
      };
      for (int qb = qb_begin; qb < qb_end; ++qb) {
        if (cls_of(qb, kb) == kEmpty) continue;
        const int slot = it % NST, phase = (it / NST) & 1;
        if (!(ok = mbar_wait(bar(Lay::B_QE + slot), phase ^ 1, abort_flag))) break;
        ++it;  // fills issued
        const uint32_t st = sbase + Lay::STAGE_OFF + slot * Lay::STAGE;
        const uint32_t fb = bar(Lay::B_QF + slot);
        if (leader) {
          mbar_arrive_expect_tx(fb, Lay::QBYTES + Lay::YBYTES + 1024);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(st + c * 16384, &p.tq, fb, 64 * c, qb * kBM, bh, keep);
          for (int c = 0; c < V / 64; ++c)
            tma_load_3d(st + Lay::QBYTES + c * 16384, &p.tdy, fb, 64 * c, qb * kBM, bh, keep);
          const size_t vo = static_cast<size_t>(bh) * p.npad + qb * kBM;
          const uint32_t vec = sbase + Lay::VEC_OFF + slot * 1024;
          bulk_load(vec, p.delta + vo, 512, fb);
          bulk_load(vec + 512, p.lse2 + vo, 512, fb);
        }
        if (t_next < 0) prefetch_next();
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
    // The last fill of each stage (iteration i = it - 1 - u fills stage i % NST).
    for (int u = 0; u < NST && u < it; ++u) {
      const int i = it - 1 - u;
      mbar_wait_inflight(bar(Lay::B_QF + i % NST), (i / NST) & 1);
    }
    if (kv_loads > 0) mbar_wait_inflight(bar(Lay::B_KV), (kv_loads - 1) & 1);
  } else if (warp == kWarpMMA) {
    const bool leader = elect_one();
    constexpr uint32_t kIdS = idesc_bf16(kBN, kBM, false, false);
    constexpr uint32_t kIdDV = idesc_bf16(kBN, V, false, true);
    constexpr uint32_t kIdDK = idesc_bf16(kBN, D, false, true);
    const uint64_t dK0 = sdesc_sw128(sbase + Lay::K_OFF, 16, 1024);
    const uint64_t dV0 = sdesc_sw128(sbase + Lay::V_OFF, 16, 1024);
    const uint64_t dSt = sdesc_sw128(sbase + Lay::STAGE_OFF, 16, 1024);     // K-major view
    const uint64_t dSm = sdesc_sw128(sbase + Lay::STAGE_OFF, 16384, 1024);  // MN-major view
    constexpr uint32_t kStage16 = Lay::STAGE >> 4, kQ16 = Lay::QBYTES >> 4;
    bool ok = true;
    // Per query block i: S^T(i) = K Q_i^T and dP^T(i) = V dY_i^T over all 128
    // queries (each product reads K or V from shared memory once), then
    // dV += P^T(i) dY_i and dK += dS^T(i) Q_i.  Issue order
    //   S(0) dP(0) | dV(0) S(1) dK(0) dP(1) | dV(1) S(2) dK(1) dP(2) | ...
    // P^T(i) sits in S^T's columns and dS^T(i) in dP^T's.  The tensor pipe runs
    // one thread's MMAs in issue order, so S(i+1) may follow dV(i), and dP(i+1)
    // may follow dK(i), without a wait.  While the elementwise warps form
    // dS(i), the pipe runs dV(i) and S(i+1); while they form P(i+1), it runs
    // dK(i) and dP(i+1).
    auto issue_s = [&](int slot) {
      const uint64_t q_k = dSt + slot * kStage16;
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_ss(tA, dK0 + off, q_k + off, kIdS, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(Lay::B_S));
      }
    };
    auto issue_dp = [&](int slot) {
      const uint64_t y_k = dSt + slot * kStage16 + kQ16;
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < V / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_ss(tB, dV0 + off, y_k + off, kIdS, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(Lay::B_DP));
      }
    };
    // acc += X^T B over the block's 128 queries, 16 per MMA: X^T (P^T or dS^T)
    // from TMEM, whose group g holds queries 32g..32g+31 as bf16 pairs in
    // columns 32g..32g+15; B (dY or Q) from the stage in its MN-major view.
    auto issue_acc = [&](uint32_t tacc, uint32_t tx, uint64_t b_m, uint32_t idesc, bool first) {
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk) {
          const uint32_t acol = 32 * (kk >> 1) + 8 * (kk & 1);
          const uint32_t rows16 = (16 * kk) * 128 >> 4;
          mma_ts(tacc, tx + acol, b_m + rows16, idesc, (!first || kk > 0) ? 1u : 0u);
        }
      }
    };
    // K and V are read by the S^T and dP^T products only: once the item's last
    // ones are issued, the commit lets the TMA warp load the next item's K and V
    // while this item's last block is still in the elementwise warps and the
    // dV, dK products.
    auto free_kv = [&]() {
      if (leader) tc_commit(bar(Lay::B_KVFREE));
    };
    int it = 0;
    for (int nitem = 0; ok; ++nitem) {
      int t;
      if (!(ok = take_item(nitem, t))) break;
      if (t < 0) break;
      int kb, bh;
      kv_item(t, nkb, p.BH, kb, bh);
      int qb_begin, qb_end;
      q_range(kb, qb_begin, qb_end);
      auto next_qb = [&](int qb) {
        for (++qb; qb < qb_end; ++qb)
          if (cls_of(qb, kb) != kEmpty) return qb;
        return qb_end;
      };
      if (!(ok = mbar_wait(bar(Lay::B_KV), nitem & 1, abort_flag))) break;
      tc_fence_after();
      int qb = next_qb(qb_begin - 1);
      int qb_n = qb < qb_end ? next_qb(qb) : qb_end;
      const int it0 = it;  // first query block of this item
      if (qb < qb_end) {
        if (!(ok = mbar_wait(bar(Lay::B_QF + it % NST), (it / NST) & 1, abort_flag))) break;
        tc_fence_after();
        issue_s(it % NST);
        issue_dp(it % NST);
      }
      if (qb_n >= qb_end) free_kv();
      while (qb < qb_end) {
        const int slot = it % NST;
        const bool more = qb_n < qb_end;
        const int qb_nn = more ? next_qb(qb_n) : qb_end;
        const int slot_n = (it + 1) % NST, phase_n = ((it + 1) / NST) & 1;
        const bool first = it == it0;
        if (!(ok = mbar_wait(bar(Lay::B_P), it & 1, abort_flag))) break;
        tc_fence_after();
        if (first && nitem > 0) {
          // dV, dK restart from zero: the previous item's epilogue has read them.
          if (!(ok = mbar_wait(bar(Lay::B_ACCFREE), (nitem - 1) & 1, abort_flag))) break;
          tc_fence_after();
        }
        issue_acc(tdV, tA, dSm + slot * kStage16 + kQ16, kIdDV, first);
        if (more) {
          if (!(ok = mbar_wait(bar(Lay::B_QF + slot_n), phase_n, abort_flag))) break;
          tc_fence_after();
          issue_s(slot_n);
        }
        if (!(ok = mbar_wait(bar(Lay::B_DSB), it & 1, abort_flag))) break;
        tc_fence_after();
        issue_acc(tdK, tB, dSm + slot * kStage16, kIdDK, first);
        if (leader) tc_commit(bar(Lay::B_QE + slot));  // Q_i, dY_i no longer read
        if (more) {
          issue_dp(slot_n);
          if (qb_nn >= qb_end) free_kv();
        }
        qb = qb_n;
        qb_n = qb_nn;
        ++it;
      }
      if (!ok) break;
      if (it == it0 && nitem > 0) {
        // An item without query blocks: keep "done" at most one phase ahead.
        if (!(ok = mbar_wait(bar(Lay::B_ACCFREE), (nitem - 1) & 1, abort_flag))) break;
      }
      if (leader) tc_commit(bar(Lay::B_DONE));  // dV, dK of the item complete
      __syncwarp();
    }
    __syncwarp();
    if (!ok && leader) {
      raise_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    if (leader) tc_commit(bar(Lay::B_DRAIN));
    mbar_wait_inflight(bar(Lay::B_DRAIN), 0);
  } else {
    // Elementwise: thread = key row r of the block; group g covers queries
    // 32g..32g+31.  Per query block two phases: P^T from S^T (then dV may
    // start), and dS^T from dP^T and the P values kept in registers.
    const int g = warp >> 2, wl = warp & 3;
    const int r = wl * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wl * 32) << 16;
    const float sl2 = p.sl2;
    int it = 0;
    bool ok = true;
    for (int nitem = 0; ok; ++nitem) {
      int t;
      if (!(ok = take_item(nitem, t))) break;
      if (t < 0) break;
      int kb, bh;
      kv_item(t, nkb, p.BH, kb, bh);
      const int k0 = kb * kBN, j = k0 + r;
      int qb_begin, qb_end;
      q_range(kb, qb_begin, qb_end);
      const int it0 = it;
      for (int qb = qb_begin; qb < qb_end; ++qb) {
        const int cls = cls_of(qb, kb);
        if (cls == kEmpty) continue;
        const int slot = it % NST;
        // Dropout: lane e draws the keep bits of query q0 + 32g + e for this warp's
        // 32 keys; the transpose gives each lane (key) its bits over the 32 queries.
        uint32_t keep = 0xFFFFFFFFu;
        if constexpr (kDrop)
          keep = transpose_bits32(keep_word32(p, bh, qb * kBM + 32 * g + lane, k0 + wl * 32), lane);
        const float* dvec = reinterpret_cast<const float*>(smem + Lay::VEC_OFF + slot * 1024);
        const float* lvec = dvec + 128;
        const int q0 = qb * kBM;
        const int cb = 32 * g;
        uint32_t allow = 0xFFFFFFFFu;
        if (cls == kPartial) {
          if (p.mask_kind == kMaskBitmask) {
            // The warp's 32 keys share one word of every bit row: lane e loads it
            // for query q0 + cb + e, and the transpose hands lane L (key j) bit L
            // of each lane's word, i.e. its keys' bits over the 32 queries.
            const int iq = q0 + cb + lane;
            const int wd = (k0 >> 5) + wl;  // == j >> 5 for every lane of the warp
            const uint32_t word = (iq < n && wd < p.words_per_row)
                                      ? __ldg(p.bits + static_cast<size_t>(iq) * p.words_per_row + wd)
                                      : 0u;
            allow = transpose_bits32(word, lane);
          }
          if (j >= nk) {
            allow = 0u;
          } else if (p.mask_kind == kMaskCausal) {
            allow = range_bits(j - off - q0 - cb, 31);
          } else if (p.mask_kind == kMaskWindow) {
            allow = range_bits(j - off - q0 - cb, j - off + p.window - 1 - q0 - cb);
          }
        }
        // The mask bits above need no product: they are formed before the wait.
        if (!(ok = mbar_wait(bar(Lay::B_S), it & 1, abort_flag))) break;
        tc_fence_after();
        float pp[32];  // p_ij of the thread's 32 queries (masked: 0), for dS
        {
          uint32_t sv[2][16];
#pragma unroll
          for (int c = 0; c < 2; ++c) tmem_ld16(tA + lane_off + cb + 16 * c, sv[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 2; ++c) reg_fence(sv[c]);
#pragma unroll
          for (int c = 0; c < 2; ++c) {  // two chunks of 16 queries
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
              const float4 l4 = *reinterpret_cast<const float4*>(lvec + cb + 16 * c + e);
              const float la[4] = {l4.x, l4.y, l4.z, l4.w};
              float pv[4];
#pragma unroll
              for (int u = 0; u < 4; u += 2) {  // query pairs: packed fp32 arithmetic
                const int q = 16 * c + e + u;
                float x0, x1;
                ffma2(x0, x1, __uint_as_float(sv[c][e + u]), __uint_as_float(sv[c][e + u + 1]),
                      sl2, sl2, -la[u], -la[u + 1]);
                pp[q] = ((allow >> q) & 1u) ? ex2(x0) : 0.f;
                pp[q + 1] = ((allow >> (q + 1)) & 1u) ? ex2(x1) : 0.f;
                if constexpr (kDrop) {
                  // Replayed mask: dV takes p xi s.
                  const float xs0 = ((keep >> q) & 1u) ? p.drop_scale : 0.f;
                  const float xs1 = ((keep >> (q + 1)) & 1u) ? p.drop_scale : 0.f;
                  fmul2(pv[u], pv[u + 1], pp[q], pp[q + 1], xs0, xs1);
                } else {
                  pv[u] = pp[q];
                  pv[u + 1] = pp[q + 1];
                }
              }
              pk[e / 2] = pack_bf16x2(pv[0], pv[1]);
              pk[e / 2 + 1] = pack_bf16x2(pv[2], pv[3]);
            }
            // P^T (bf16 pairs) over the first 16 columns of this group's range.
            tmem_st8(tA + lane_off + cb + 8 * c, pk);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(Lay::B_P));
        }
        if (!(ok = mbar_wait(bar(Lay::B_DP), it & 1, abort_flag))) break;
        tc_fence_after();
        {
          uint32_t dpv[2][16];
#pragma unroll
          for (int c = 0; c < 2; ++c) tmem_ld16(tB + lane_off + cb + 16 * c, dpv[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 2; ++c) reg_fence(dpv[c]);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t dk[8];
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
              const float4 d4 = *reinterpret_cast<const float4*>(dvec + cb + 16 * c + e);
              const float da[4] = {d4.x, d4.y, d4.z, d4.w};
              float gv[4];
#pragma unroll
              for (int u = 0; u < 4; u += 2) {
                const int q = 16 * c + e + u;
                float dq0 = __uint_as_float(dpv[c][e + u]), dq1 = __uint_as_float(dpv[c][e + u + 1]);
                if constexpr (kDrop) {
                  // Replayed mask: dP = xi s (G_i . V_j).
                  const float xs0 = ((keep >> q) & 1u) ? p.drop_scale : 0.f;
                  const float xs1 = ((keep >> (q + 1)) & 1u) ? p.drop_scale : 0.f;
                  fmul2(dq0, dq1, dq0, dq1, xs0, xs1);
                }
                float t0, t1;
                fadd2(t0, t1, dq0, dq1, -da[u], -da[u + 1]);
                fmul2(gv[u], gv[u + 1], pp[q], pp[q + 1], t0, t1);
              }
              dk[e / 2] = pack_bf16x2(gv[0], gv[1]);
              dk[e / 2 + 1] = pack_bf16x2(gv[2], gv[3]);
            }
            // dS^T (bf16 pairs) over the first 16 columns of this group's range.
            tmem_st8(tB + lane_off + cb + 8 * c, dk);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(Lay::B_DSB));
        }
        ++it;
      }
      if (!ok) break;
      // Epilogue.  Every group reads its D/2 columns of dV (g = 0, 1) or dK
      // (g = 2, 3; scaled by c) and releases the accumulators at once.  The
      // rows then leave through one shared-memory tile in the TMA layout
      // (64-column boxes, 128-byte swizzle) and TMA stores, which write whole
      // lines and clip rows past nk: dV first, then dK in the same tile.
      if (!(ok = mbar_wait(bar(Lay::B_DONE), nitem & 1, abort_flag))) break;
      tc_fence_after();
      constexpr int HC = D / 2;  // columns per group (D == V)
      const bool is_dv = g < 2;
      const int c0 = (g & 1) * HC;
      uint32_t pk[HC / 2];
      {
        uint32_t o[HC / 16][16];
        if (it > it0) {
#pragma unroll
          for (int c = 0; c < HC / 16; ++c)
            tmem_ld16((is_dv ? tdV : tdK) + lane_off + c0 + 16 * c, o[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < HC / 16; ++c) reg_fence(o[c]);
        } else {
#pragma unroll
          for (int c = 0; c < HC / 16; ++c)
#pragma unroll
            for (int e = 0; e < 16; ++e) o[c][e] = 0u;
        }
        const float mul = is_dv ? 1.f : p.scale;
#pragma unroll
        for (int e = 0; e < HC / 2; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(o[e >> 3][(2 * e) & 15]) * mul,
                              __uint_as_float(o[e >> 3][(2 * e + 1) & 15]) * mul);
      }
      tc_fence_before();
      mbar_arrive(bar(Lay::B_ACCFREE));  // dV, dK read: the next item may restart them
      if (warp == kEwWarps / 2) {
        // Issuer of the dK stores (thread 256): the previous item's have read the tile.
        if (lane == 0) {
          bulk_wait_read_all();
          mbar_arrive(bar(Lay::B_EPIFV));
        }
        __syncwarp();
      }
      if (!(ok = mbar_wait(bar(is_dv ? Lay::B_EPIFV : Lay::B_EPIFK), nitem & 1, abort_flag))) break;
      const uint32_t tile = sbase + Lay::EPI_OFF;
#pragma unroll
      for (int u = 0; u < HC / 8; ++u) {
        const int col = c0 + 8 * u;
        const uint32_t addr = tile + (col >> 6) * (kBN * 128) + r * 128 +
                              ((((col & 63) >> 3) ^ (r & 7)) << 4);
        st_shared_v4(addr, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(is_dv ? Lay::B_EPIV : Lay::B_EPIK));
      if (threadIdx.x == (is_dv ? 0 : 32 * (kEwWarps / 2))) {
        if (mbar_wait(bar(is_dv ? Lay::B_EPIV : Lay::B_EPIK), nitem & 1, abort_flag)) {
          const CUtensorMap* map = is_dv ? &p.tdv : &p.tdk;
          const int cols = is_dv ? p.v : p.d;  // no box that starts past the columns
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            if (64 * c < cols) tma_store_3d(map, tile + c * (kBN * 128), 64 * c, k0, bh);
          bulk_commit();
          if (is_dv) {
            bulk_wait_read_all();
            mbar_arrive(bar(Lay::B_EPIFK));
          }
        } else {
          ok = false;
        }
      }
      ok = __all_sync(0xFFFFFFFFu, ok);
    }
    if (!ok) {
      raise_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    // The stores' issuers: all of their stores complete before the CTA ends.
    if (threadIdx.x == 0 || threadIdx.x == 32 * (kEwWarps / 2)) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// =========================================================================
// Query-major kernel: dQ (and delta)
// =========================================================================
template <int D, int V>
struct QLayout {
  static constexpr int QBYTES = kBM * D * 2;
  static constexpr int YBYTES = kBM * V * 2;
  static constexpr int KBYTES = kBN * D * 2;
  static constexpr int VBYTES = kBN * V * 2;
  static constexpr int SLOT = KBYTES > VBYTES ? KBYTES : VBYTES;
  // Two rings over one slot array: K tiles in slots [0, NK), V tiles in
  // [NK, NK + NV).  K(t) is read until dQ(t) completes, V(t) only until dP(t)
  // does, so K gets the deeper ring: its refill then has a whole step.
  static constexpr int NK = D == 128 ? 3 : 5;
  static constexpr int NV = D == 128 ? 1 : 3;
  static constexpr int NS = NK + NV;
  static constexpr int Q_OFF = 0;
  static constexpr int Y_OFF = QBYTES;
  static constexpr int SLOT_OFF = Y_OFF + YBYTES;
  // Epilogue tile: kBM rows of dQ as 64-column boxes (128-byte swizzle).
  static constexpr int EPI_OFF = SLOT_OFF + NS * SLOT;
  // Partial sums of delta_i = dY_i . Y_i, one per elementwise group and row.
  static constexpr int PART_OFF = EPI_OFF + kBM * D * 2;
  static constexpr int BAR_OFF = PART_OFF + 4 * kBM * 4;
  static constexpr int B_Q = 0, B_QFREE = 1, B_KVF = 2, B_KVE = B_KVF + NS, B_SDP = B_KVE + NS,
                       B_DS = B_SDP + 1, B_SFREE = B_DS + 2, B_DONE = B_SFREE + 1,
                       B_DREAD = B_DONE + 1, B_ITEMF = B_DREAD + 1, B_ITEME = B_ITEMF + 2,
                       B_EPIF = B_ITEME + 2, B_EPI = B_EPIF + 1, B_DPART = B_EPI + 1,
                       B_DRAIN = B_DPART + 1, NBAR = B_DRAIN + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int CLS_OFF = MISC_OFF + 16;
  static constexpr int TOTAL = CLS_OFF + 2 * (kMaxBlocks / 32) * 4;
  static_assert(TOTAL <= 232448, "shared memory");
};

template <int D, int V, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_q_kernel(const __grid_constant__ Bwd2Params p) {
  using Lay = QLayout<D, V>;
  constexpr int NS = Lay::NS;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + Lay::BAR_OFF;
  auto bar = [&](int k) { return bar0 + 8u * k; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* item_ring = reinterpret_cast<volatile int*>(misc + 2);  // two entries
  uint32_t* anyb = reinterpret_cast<uint32_t*>(smem + Lay::CLS_OFF);
  uint32_t* notallb = anyb + kMaxBlocks / 32;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.n, nk = p.nk, off = p.off;
  const int nqb = (n + kBM - 1) / kBM, nkb = (nk + kBN - 1) / kBN;
  const int items = nqb * p.BH;
  // Persistent: as in the dK/dV kernel, the TMA warp takes items from a
  // counter and hands them out through a two-entry ring; item t is
  // (query block nqb - 1 - x, slice bh) with (x, bh) = kv_item(t): heaviest
  // (causal) query blocks first inside each group of slices.
  auto item_of = [&](int t, int& qb, int& bh) {
    int x;
    kv_item(t, nqb, p.BH, x, bh);
    qb = nqb - 1 - x;
  };
  // Key blocks that rows q0..q1 (at absolute positions q0 + off ..) can reach.
  auto kb_range = [&](int qb, int& kb_begin, int& kb_end) {
    const int q0 = qb * kBM, q1 = min(q0 + kBM, n) - 1;
    kb_begin = 0;
    kb_end = nkb;
    if (p.mask_kind == kMaskCausal || p.mask_kind == kMaskWindow)
      kb_end = q1 + off < 0 ? 0 : min(nkb, (q1 + off) / kBN + 1);
    if (p.mask_kind == kMaskWindow) kb_begin = min(kb_end, max(0, q0 + off - p.window + 1) / kBN);
  };

  if ((sbase & 1023u) != 0u) {
    if (threadIdx.x == 0) raise_status(p.status, kStatusTimeout);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(bar(Lay::B_Q), 1);
    mbar_init(bar(Lay::B_QFREE), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(Lay::B_KVF + s), 1);
      mbar_init(bar(Lay::B_KVE + s), 1);
    }
    mbar_init(bar(Lay::B_SDP), 1);
    // dS(t) written: one barrier per block parity.  dS(t + 2) needs S(t + 2),
    // which the MMA warp issues only after its wait for dS(t), so neither
    // barrier ever runs a phase ahead of that wait; with one barrier the
    // elementwise warps could complete dS(t) and dS(t + 1) before it.
    mbar_init(bar(Lay::B_DS + 0), kEwWarps * 32);
    mbar_init(bar(Lay::B_DS + 1), kEwWarps * 32);
    mbar_init(bar(Lay::B_SFREE), kEwWarps * 32);
    mbar_init(bar(Lay::B_DONE), 1);
    mbar_init(bar(Lay::B_DREAD), kEwWarps * 32);  // the epilogue has read dQ
    for (int e = 0; e < 2; ++e) {
      mbar_init(bar(Lay::B_ITEMF + e), 1);
      mbar_init(bar(Lay::B_ITEME + e), 1 + kEwWarps);  // MMA warp + elementwise warps
    }
    mbar_init(bar(Lay::B_EPIF), 1);  // the previous item's dQ stores have read the tile
    mbar_init(bar(Lay::B_EPI), kEwWarps * 32);
    mbar_init(bar(Lay::B_DPART), kEwWarps * 32);  // delta partial sums written (dY read)
    mbar_init(bar(Lay::B_DRAIN), 1);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(sbase + Lay::MISC_OFF, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  if (threadIdx.x < 2 * (kMaxBlocks / 32)) anyb[threadIdx.x] = 0u;
  __syncthreads();
  if (p.mask_kind == kMaskBitmask) {
    // The tile table is per query block: the launcher gives every CTA exactly
    // one item for this mask kind (item blockIdx.x).
    int qb0, bh0, kb_begin, kb_end;
    item_of(blockIdx.x, qb0, bh0);
    kb_range(qb0, kb_begin, kb_end);
    build_bitmask_table(p, false, qb0, kb_begin, kb_end, anyb, notallb);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const uint32_t tS = tmem, tD0 = tmem + 128, tQ = tmem + 384;
  auto cls_of = [&](int qb, int kb) {
    return classify_tile(p, qb, kb, (anyb[kb >> 5] >> (kb & 31)) & 1u,
                         (notallb[kb >> 5] >> (kb & 31)) & 1u);
  };
  // Consumers: item nitem from the ring (waits for it, then frees the entry).
  auto take_item = [&](int nitem, int& t) {
    const int e = nitem & 1;
    if (!mbar_wait(bar(Lay::B_ITEMF + e), (nitem >> 1) & 1, abort_flag)) return false;
    t = item_ring[e];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(Lay::B_ITEME + e));
    return true;
  };

  if (warp == kWarpTMA) {
    const bool leader = elect_one();
    if (leader) {
      prefetch_tmap(&p.tq);
      prefetch_tmap(&p.tk);
      prefetch_tmap(&p.tv);
      prefetch_tmap(&p.tdy);
      prefetch_tmap(&p.tdq);
      prefetch_tmap(&p.ty);
    }
    const uint64_t keep = policy_evict_last(), stream = policy_evict_first();
    int it = 0, q_loads = 0, k_fills = 0, v_fills = 0;  // blocks; copies issued
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
      if (lane == 0) claimed = atomicAdd(p.sched + 1, 1u);
      int qb, bh, kb_begin, kb_end;
      item_of(t, qb, bh);
      kb_range(qb, kb_begin, kb_end);
      const int q0 = qb * kBM;
      // Q and dY of the item once the previous item's S, dP products no longer read them.
      if (nitem > 0 && !(ok = mbar_wait(bar(Lay::B_QFREE), (nitem - 1) & 1, abort_flag))) break;
      if (leader) {
        mbar_arrive_expect_tx(bar(Lay::B_Q), Lay::QBYTES + Lay::YBYTES);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sbase + Lay::Q_OFF + c * 16384, &p.tq, bar(Lay::B_Q), 64 * c, q0, bh, stream);
        for (int c = 0; c < V / 64; ++c)
          tma_load_3d(sbase + Lay::Y_OFF + c * 16384, &p.tdy, bar(Lay::B_Q), 64 * c, q0, bh, stream);
      }
      ++q_loads;
      // The next item's Q and dY go into L2 after this item's first block.
      int t_next = -1;
      auto prefetch_next = [&]() {
        t_next = static_cast<int>(
            min(__shfl_sync(0xFFFFFFFFu, claimed, 0) + gridDim.x, static_cast<unsigned>(items)));
        if (t_next < items && leader) {
          int qbn, bhn;
          item_of(t_next, qbn, bhn);
          for (int c = 0; c < D / 64; ++c)
            if (64 * c < p.d) tma_prefetch_3d(&p.tq, 64 * c, qbn * kBM, bhn);
          for (int c = 0; c < V / 64; ++c) {
            if (64 * c >= p.v) break;
            tma_prefetch_3d(&p.tdy, 64 * c, qbn * kBM, bhn);
            tma_prefetch_3d(&p.ty, 64 * c, qbn * kBM, bhn);  // for delta
          }
        }
      };
      for (int kb = kb_begin; kb < kb_end && ok; ++kb) {
        if (cls_of(qb, kb) == kEmpty) continue;
        // Block it: V(it) into slot NK + it % NV, then K(it) into slot it % NK.
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          const int slot = kv == 0 ? Lay::NK + it % Lay::NV : it % Lay::NK;
          const int phase = kv == 0 ? (it / Lay::NV) & 1 : (it / Lay::NK) & 1;
          if (!mbar_wait(bar(Lay::B_KVE + slot), phase ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t dst = sbase + Lay::SLOT_OFF + slot * Lay::SLOT;
          if (leader) {
            if (kv == 1) {
              mbar_arrive_expect_tx(bar(Lay::B_KVF + slot), Lay::KBYTES);
              for (int c = 0; c < D / 64; ++c)
                tma_load_3d(dst + c * 16384, &p.tk, bar(Lay::B_KVF + slot), 64 * c, kb * kBN, bh,
                            keep);
            } else {
              mbar_arrive_expect_tx(bar(Lay::B_KVF + slot), Lay::VBYTES);
              for (int c = 0; c < V / 64; ++c)
                tma_load_3d(dst + c * 16384, &p.tv, bar(Lay::B_KVF + slot), 64 * c, kb * kBN, bh,
                            keep);
            }
          }
          ++(kv == 0 ? v_fills : k_fills);
        }
        ++it;
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
    // Never leave with copies in flight: the last fill of every slot (the i-th
    // K copy went to slot i % NK, the i-th V copy to slot NK + i % NV) and the
    // last Q, dY.
    for (int u = 0; u < Lay::NK && u < k_fills; ++u) {
      const int i = k_fills - 1 - u;
      mbar_wait_inflight(bar(Lay::B_KVF + i % Lay::NK), (i / Lay::NK) & 1);
    }
    for (int u = 0; u < Lay::NV && u < v_fills; ++u) {
      const int i = v_fills - 1 - u;
      mbar_wait_inflight(bar(Lay::B_KVF + Lay::NK + i % Lay::NV), (i / Lay::NV) & 1);
    }
    if (q_loads > 0) mbar_wait_inflight(bar(Lay::B_Q), (q_loads - 1) & 1);
  } else if (warp == kWarpMMA) {
    const bool leader = elect_one();
    constexpr uint32_t kIdSS = idesc_bf16(kBM, kBN, false, false);
    constexpr uint32_t kIdDQ = idesc_bf16(kBM, D, false, true);
    const uint64_t dQk = sdesc_sw128(sbase + Lay::Q_OFF, 16, 1024);
    const uint64_t dYk = sdesc_sw128(sbase + Lay::Y_OFF, 16, 1024);
    const uint64_t dSk = sdesc_sw128(sbase + Lay::SLOT_OFF, 16, 1024);
    const uint64_t dSm = sdesc_sw128(sbase + Lay::SLOT_OFF, 16384, 1024);
    constexpr uint32_t kSlot16 = Lay::SLOT >> 4;
    bool ok = true;
    // Block t (counted across items) uses K slot t % NK and V slot NK + t % NV.
    auto issue_dp = [&](int tt) {
      const int vs = Lay::NK + tt % Lay::NV;
      const uint32_t tD = tD0 + 128 * (tt & 1);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < V / 16; ++kk) {
          const uint32_t o16 = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_ss(tD, dYk + o16, dSk + vs * kSlot16 + o16, kIdSS, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(Lay::B_KVE + vs));  // V(t) is no longer needed once dP(t) is done
      }
    };
    auto issue_s = [&](int tt) {
      const int ks = tt % Lay::NK;
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o16 = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_ss(tS, dQk + o16, dSk + ks * kSlot16 + o16, kIdSS, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(Lay::B_SDP));
      }
    };
    auto v_full = [&](int tt) {
      return mbar_wait(bar(Lay::B_KVF + Lay::NK + tt % Lay::NV), (tt / Lay::NV) & 1, abort_flag);
    };
    auto k_full = [&](int tt) {
      return mbar_wait(bar(Lay::B_KVF + tt % Lay::NK), (tt / Lay::NK) & 1, abort_flag);
    };
    int t = 0, ne = 0;  // ne: items with key blocks so far (phases of B_DPART)
    for (int nitem = 0; ok; ++nitem) {
      int ti;
      if (!(ok = take_item(nitem, ti))) break;
      if (ti < 0) break;
      int qb, bh, kb_begin, kb_end;
      item_of(ti, qb, bh);
      kb_range(qb, kb_begin, kb_end);
      (void)bh;
      // Compact list of the key blocks to visit: recomputed on the fly.
      auto next_kb = [&](int kb) {
        for (++kb; kb < kb_end; ++kb)
          if (cls_of(qb, kb) != kEmpty) return kb;
        return kb_end;
      };
      if (!(ok = mbar_wait(bar(Lay::B_Q), nitem & 1, abort_flag))) break;
      tc_fence_after();
      int kb = next_kb(kb_begin - 1);
      int kb_n = kb < kb_end ? next_kb(kb) : kb_end;
      const int t0 = t;
      // Q and dY are read by the S and dP products and, for delta, by the
      // elementwise warps of an item with key blocks.
      const bool nonempty = kb < kb_end;
      auto free_q = [&]() {
        if (nonempty && !mbar_wait(bar(Lay::B_DPART), ne & 1, abort_flag)) return false;
        if (leader) tc_commit(bar(Lay::B_QFREE));
        return true;
      };
      // Prologue: dP(t0) -> its buffer, S(t0) -> S once the previous item's
      // last S is in the elementwise warps' registers.
      if (kb < kb_end) {
        if (!(ok = v_full(t))) break;
        tc_fence_after();
        issue_dp(t);
        if (t > 0 && !(ok = mbar_wait(bar(Lay::B_SFREE), (t - 1) & 1, abort_flag))) break;
        if (!(ok = k_full(t))) break;
        tc_fence_after();
        issue_s(t);
      }
      if (kb_n >= kb_end && !(ok = free_q())) break;
      while (kb < kb_end) {
        const bool more = kb_n < kb_end;
        const int kb_nn = more ? next_kb(kb_n) : kb_end;
        if (more) {
          // dP(t+1) -> the other buffer (its dS(t-1) was read by dQ(t-1), issued earlier).
          if (!(ok = v_full(t + 1))) break;
          tc_fence_after();
          issue_dp(t + 1);
          // S(t+1) as soon as the elementwise warps hold S(t) in registers.
          if (!(ok = mbar_wait(bar(Lay::B_SFREE), t & 1, abort_flag))) break;
          if (!(ok = k_full(t + 1))) break;
          tc_fence_after();
          issue_s(t + 1);
          if (kb_nn >= kb_end && !(ok = free_q())) break;
        }
        if (!(ok = mbar_wait(bar(Lay::B_DS + (t & 1)), (t >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        // dQ += dS(t) K_t  (A = dS bf16 in TMEM over dP(t), keys packed; B = K_t MN-major)
        const int ks = t % Lay::NK;
        const uint32_t tD = tD0 + 128 * (t & 1);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts(tQ, tD + 32 * (kk >> 1) + 8 * (kk & 1), dSm + ks * kSlot16 + kk * 128, kIdDQ,
                   (t > t0 || kk > 0) ? 1u : 0u);
          tc_commit(bar(Lay::B_KVE + ks));
        }
        kb = kb_n;
        kb_n = kb_nn;
        ++t;
      }
      if (!ok) break;
      if (nonempty) ++ne;
      // "dQ done" stays at most one phase ahead of the epilogue, also through
      // items without key blocks.
      if (nitem > 0 && !(ok = mbar_wait(bar(Lay::B_DREAD), (nitem - 1) & 1, abort_flag))) break;
      if (leader) tc_commit(bar(Lay::B_DONE));
      __syncwarp();
    }
    __syncwarp();
    if (!ok && leader) {
      raise_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    if (leader) tc_commit(bar(Lay::B_DRAIN));
    mbar_wait_inflight(bar(Lay::B_DRAIN), 0);
  } else {
    // Elementwise: thread = query row r; group g covers keys 32g..32g+31.
    const int g = warp >> 2, wl = warp & 3;
    const int r = wl * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wl * 32) << 16;
    const float sl2 = p.sl2;
    float* part = reinterpret_cast<float*>(smem + Lay::PART_OFF);  // [4][kBM]
    int t = 0, ne = 0;  // ne: items with key blocks so far (phases of B_DPART)
    bool ok = true;
    // Y_i (this group's V/4 columns) and L_i of an item's row r, loaded as soon
    // as the item is known: for the next item that is before this item's
    // epilogue, so the loads overlap it.
    constexpr int CV = V / 4;
    uint4 yv[CV / 8];
    float Li = -INFINITY;
    auto load_row = [&](int tix) {
      int qbx, bhx;
      item_of(tix, qbx, bhx);
      const int ix = qbx * kBM + r;
      Li = -INFINITY;
      if (ix < n) {
        const uint4* yrow = reinterpret_cast<const uint4*>(
            p.Y + (static_cast<size_t>(bhx) * n + ix) * p.v + CV * g);
#pragma unroll
        for (int u = 0; u < CV / 8; ++u)  // columns past v: zero (as in the staged dY)
          yv[u] = CV * g + 8 * u < p.v ? __ldg(yrow + u) : make_uint4(0u, 0u, 0u, 0u);
        Li = __ldg(p.L + static_cast<size_t>(bhx) * n + ix);
      }
    };
    int ti = -1;
    if ((ok = take_item(0, ti)) && ti >= 0) load_row(ti);
    for (int nitem = 0; ok && ti >= 0; ++nitem) {
      int qb, bh, kb_begin, kb_end;
      item_of(ti, qb, bh);
      kb_range(qb, kb_begin, kb_end);
      const int q0 = qb * kBM;
      const int i = q0 + r;
      const size_t vo = static_cast<size_t>(bh) * p.npad + q0 + r;
      // A row whose L is -inf had an empty allowed set: p = 0 below, and the
      // status word says so.
      if (g == 0 && i < n && Li == -INFINITY) raise_status(p.status, kStatusEmptyRow);
      // delta_i = dY_i . Y_i ("Exact tiled softmax attention ...", Reverse
      // procedure) and L_i log2(e) for this query block: group g sums columns
      // V/4 g .. of dY (from the staged tile) times Y, the four partial sums
      // meet in shared memory.  Both go to the workspace for the dK/dV kernel,
      // which runs after this one.  Padding rows: delta 0, L log2(e) = +inf.
      int kb_first = kb_begin;
      while (kb_first < kb_end && cls_of(qb, kb_first) == kEmpty) ++kb_first;
      float lse2 = INFINITY, dl = 0.f;
      if (kb_first < kb_end) {
        if (!(ok = mbar_wait(bar(Lay::B_Q), nitem & 1, abort_flag))) break;
        float acc = 0.f;
        if (i < n) {
#pragma unroll
          for (int u = 0; u < CV / 8; ++u) {
            const int col = CV * g + 8 * u;
            const uint4 gv = ld_shared_v4(sbase + Lay::Y_OFF + (col >> 6) * 16384 + r * 128 +
                                          ((((col & 63) >> 3) ^ (r & 7)) << 4));
            const uint32_t ya[4] = {yv[u].x, yv[u].y, yv[u].z, yv[u].w};
            const uint32_t ga[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc = fmaf(__uint_as_float(ya[e] << 16), __uint_as_float(ga[e] << 16), acc);
              acc = fmaf(__uint_as_float(ya[e] & 0xFFFF0000u), __uint_as_float(ga[e] & 0xFFFF0000u),
                         acc);
            }
          }
        }
        part[g * kBM + r] = acc;
        mbar_arrive(bar(Lay::B_DPART));
        if (!(ok = mbar_wait(bar(Lay::B_DPART), ne & 1, abort_flag))) break;
        ++ne;
        if (i < n) {
          dl = (part[r] + part[kBM + r]) + (part[2 * kBM + r] + part[3 * kBM + r]);
          lse2 = Li == -INFINITY ? INFINITY : Li * kLog2e;  // p = 0 on empty rows
        }
      }
      if (g == 0) {
        p.delta[vo] = dl;
        p.lse2[vo] = lse2;
      }
      const int t0 = t;
      for (int kb = kb_begin; kb < kb_end; ++kb) {
        const int cls = cls_of(qb, kb);
        if (cls == kEmpty) continue;
        const int kc = kb * kBN + 32 * g;  // first key of this group
        // A bit-row word is loaded before the wait for S and dP, so that the
        // load is in flight meanwhile.
        uint32_t bitw = 0xFFFFFFFFu;
        if (p.mask_kind == kMaskBitmask && cls == kPartial) {
          const int w = kb * 4 + g;
          bitw = (i < n && w < p.words_per_row)
                     ? __ldg(p.bits + static_cast<size_t>(i) * p.words_per_row + w)
                     : 0u;
        }
        if (!(ok = mbar_wait(bar(Lay::B_SDP), t & 1, abort_flag))) break;
        tc_fence_after();
        uint32_t allow = 0xFFFFFFFFu;
        if (cls == kPartial) {
          int lo = 0, hi = nk - 1;
          if (p.mask_kind == kMaskCausal || p.mask_kind == kMaskWindow) hi = min(hi, i + off);
          if (p.mask_kind == kMaskWindow) lo = max(lo, i + off - p.window + 1);
          allow = range_bits(lo - kc, hi - kc) & bitw;
        }
        const uint32_t tD = tD0 + 128 * (t & 1) + lane_off;
        uint32_t sv[2][16], dpv[2][16];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          tmem_ld16(tS + lane_off + 32 * g + 16 * c, sv[c]);
          tmem_ld16(tD + 32 * g + 16 * c, dpv[c]);
        }
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          reg_fence(sv[c]);
          reg_fence(dpv[c]);
        }
        // S(t) is in registers: the MMA warp may overwrite it with S(t+1).
        tc_fence_before();
        mbar_arrive(bar(Lay::B_SFREE));
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint32_t (&s)[16] = sv[c];
          const uint32_t (&dp)[16] = dpv[c];
          uint32_t dk[8];
          uint4 rw;  // dropout: Philox words of keys kc + 16c + 8*(e/8) .. of row i
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            float x0, x1;  // packed fp32 arithmetic over the key pair
            ffma2(x0, x1, __uint_as_float(s[e]), __uint_as_float(s[e + 1]), sl2, sl2, -lse2,
                  -lse2);
            float p0 = ex2(x0);
            float p1 = ex2(x1);
            if (!((allow >> (16 * c + e)) & 1u)) p0 = 0.f;
            if (!((allow >> (16 * c + e + 1)) & 1u)) p1 = 0.f;
            float dp0 = __uint_as_float(dp[e]), dp1 = __uint_as_float(dp[e + 1]);
            if constexpr (kDrop) {
              // Replayed mask: dP = xi s (G_i . V_j); keys e, e+1 share one word.
              if ((e & 7) == 0)
                rw = keep_words(p.seed_lo, p.seed_hi, bh, i, (kc + 16 * c + e) >> 3);
              const int wi = (e & 7) >> 1;
              const uint32_t w = wi == 0 ? rw.x : wi == 1 ? rw.y : wi == 2 ? rw.z : rw.w;
              dp0 *= (w & 0xFFFFu) >= p.drop_t ? p.drop_scale : 0.f;
              dp1 *= w >= (p.drop_t << 16) ? p.drop_scale : 0.f;
            }
            float t0f, t1f, g0, g1;
            fadd2(t0f, t1f, dp0, dp1, -dl, -dl);
            fmul2(g0, g1, p0, p1, t0f, t1f);
            dk[e / 2] = pack_bf16x2(g0, g1);
          }
          tmem_st8(tD + 32 * g + 8 * c, dk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(Lay::B_DS + (t & 1)));
        ++t;
      }
      if (!ok) break;
      // The next item now (the ring holds it by the time this item's blocks are
      // done): its row loads overlap this item's epilogue.
      int tn = -1;
      if (!(ok = take_item(nitem + 1, tn))) break;
      if (tn >= 0) load_row(tn);
      // Epilogue: dQ_i = c * acc, bf16; group g reads columns CW g .. CW g + CW - 1,
      // releases the accumulator, and the rows leave through one shared-memory
      // tile in the TMA layout (64-column boxes, 128-byte swizzle) and TMA
      // stores, which write whole lines and clip rows past n.
      if (!(ok = mbar_wait(bar(Lay::B_DONE), nitem & 1, abort_flag))) break;
      tc_fence_after();
      constexpr int CW = D / 4;  // columns per group
      uint32_t pk[CW / 2];
      {
        uint32_t o[CW / 16][16];
        if (t > t0) {
#pragma unroll
          for (int ch = 0; ch < CW / 16; ++ch) tmem_ld16(tQ + lane_off + CW * g + 16 * ch, o[ch]);
          tmem_ld_wait();
#pragma unroll
          for (int ch = 0; ch < CW / 16; ++ch) reg_fence(o[ch]);
        } else {
#pragma unroll
          for (int ch = 0; ch < CW / 16; ++ch)
#pragma unroll
            for (int e = 0; e < 16; ++e) o[ch][e] = 0u;
        }
#pragma unroll
        for (int e = 0; e < CW / 2; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(o[e >> 3][(2 * e) & 15]) * p.scale,
                              __uint_as_float(o[e >> 3][(2 * e + 1) & 15]) * p.scale);
      }
      tc_fence_before();
      mbar_arrive(bar(Lay::B_DREAD));  // the next item's first dQ product may overwrite it
      if (threadIdx.x == 0) {
        bulk_wait_read_all();
        mbar_arrive(bar(Lay::B_EPIF));
      }
      if (!(ok = mbar_wait(bar(Lay::B_EPIF), nitem & 1, abort_flag))) break;
      const uint32_t tile = sbase + Lay::EPI_OFF;
#pragma unroll
      for (int u = 0; u < CW / 8; ++u) {
        const int col = CW * g + 8 * u;
        const uint32_t addr = tile + (col >> 6) * (kBM * 128) + r * 128 +
                              ((((col & 63) >> 3) ^ (r & 7)) << 4);
        st_shared_v4(addr, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(Lay::B_EPI));
      if (threadIdx.x == 0) {
        if (mbar_wait(bar(Lay::B_EPI), nitem & 1, abort_flag)) {
#pragma unroll
          for (int c = 0; c < D / 64; ++c)  // no box that starts past dQ's columns
            if (64 * c < p.d) tma_store_3d(&p.tdq, tile + c * (kBM * 128), 64 * c, q0, bh);
          bulk_commit();
        } else {
          ok = false;
        }
      }
      ok = __all_sync(0xFFFFFFFFu, ok);
      ti = tn;
    }
    if (!ok) {
      raise_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    // The stores' issuer: all of its stores complete before the CTA ends.
    if (threadIdx.x == 0) bulk_wait_all();
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
cudaError_t launch_split(const BwdArgs& a, cudaStream_t s) {
  const Problem& pr = a.p;
  Bwd2Params p;
  // Tensor maps of the true widths: loads fill the columns up to D with zeros
  // (no contribution to S, dP, dV or dK), stores clip them.
  if (!make_tmap_bf16(&p.tq, a.Q, pr.d, pr.n, pr.BH) ||
      !make_tmap_bf16(&p.tk, a.K, pr.d, pr.nk, pr.BH) ||
      !make_tmap_bf16(&p.tv, a.V, pr.v, pr.nk, pr.BH) ||
      !make_tmap_bf16(&p.tdy, a.dY, pr.v, pr.n, pr.BH) ||
      !make_tmap_bf16(&p.tdk, a.dK, pr.d, pr.nk, pr.BH) ||
      !make_tmap_bf16(&p.tdv, a.dV, pr.v, pr.nk, pr.BH) ||
      !make_tmap_bf16(&p.tdq, a.dQ, pr.d, pr.n, pr.BH) ||
      !make_tmap_bf16(&p.ty, a.Y, pr.v, pr.n, pr.BH))
    return cudaErrorInvalidValue;
  p.n = pr.n;
  p.nk = pr.nk;
  p.off = pr.nk - pr.n;
  p.npad = a.npad;
  p.d = pr.d;
  p.v = pr.v;
  p.BH = pr.BH;
  p.mask_kind = pr.mask_kind;
  p.window = pr.window;
  p.words_per_row = pr.words_per_row;
  p.bits = pr.bitmask;
  p.delta = a.delta;
  p.lse2 = a.lse2;
  p.Y = static_cast<const __nv_bfloat16*>(a.Y);
  p.L = a.L;
  p.sl2 = pr.scale * kLog2e;
  p.scale = pr.scale;
  p.dQ = static_cast<__nv_bfloat16*>(a.dQ);
  p.dK = static_cast<__nv_bfloat16*>(a.dK);
  p.dV = static_cast<__nv_bfloat16*>(a.dV);
  p.status = a.status;
  p.sched = a.status + kSchedWord;
  p.drop_t = pr.drop_t;
  p.seed_lo = pr.seed_lo;
  p.seed_hi = pr.seed_hi;
  p.drop_scale = pr.drop_scale;
  const bool drop = pr.drop_t != 0;
  auto kv = drop ? tc_bwd_kv_kernel<D, D, true> : tc_bwd_kv_kernel<D, D, false>;
  auto qk = drop ? tc_bwd_q_kernel<D, D, true> : tc_bwd_q_kernel<D, D, false>;
  cudaError_t e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       KvLayout<D, D>::TOTAL);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(qk, cudaFuncAttributeMaxDynamicSharedMemorySize, QLayout<D, D>::TOTAL);
  if (e != cudaSuccess) {
    record_error("tc_bwd2: cudaFuncSetAttribute", static_cast<int>(e), cudaGetErrorString(e));
    return e;
  }
  const int nkb = (pr.nk + kBN - 1) / kBN, nqb = (pr.n + kBM - 1) / kBM;
  before_launch(kKernBwd, s);
  // Persistent kernels: one CTA per SM, items handed out by a counter; one
  // item per CTA for the bitmask, whose tile table each CTA builds once.
  int sms = 148;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  }
  auto grid_of = [&](int items) {
    return pr.mask_kind == kMaskBitmask || items < sms ? items : sms;
  };
  // The dQ kernel first: it also forms delta and L log2(e), which the dK/dV
  // kernel reads.
  before_launch(kKernBwdQ, s);
  qk<<<grid_of(nqb * pr.BH), kThreads, QLayout<D, D>::TOTAL, s>>>(p);
  e = cudaGetLastError();
  after_launch(kKernBwdQ, s);
  if (e == cudaSuccess) {
    kv<<<grid_of(nkb * pr.BH), kThreads, KvLayout<D, D>::TOTAL, s>>>(p);
    e = cudaGetLastError();
  }
  after_launch(kKernBwd, s);
  return e;
}

}  // namespace

// Widths up to 128 in steps of 8 run on the kernels of width 64 or 128 (see
// the tensor maps in launch_split).
bool tc_bwd_split_supported(const Problem& p) {
  if (p.dtype != kBF16 || p.d < 8 || p.v < 8 || p.d > 128 || p.v > 128 || p.d % 8 != 0 ||
      p.v % 8 != 0)
    return false;
  if (p.mask_kind == kMaskBitmask && (p.n > kMaxBlocks * kBM || p.nk > kMaxBlocks * kBN))
    return false;
  return tmap_encoder_available();
}

cudaError_t launch_tc_bwd_split(const BwdArgs& a, cudaStream_t s) {
  return a.p.d <= 64 && a.p.v <= 64 ? launch_split<64>(a, s) : launch_split<128>(a, s);
}

}  // namespace exattn
