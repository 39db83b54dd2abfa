// Reverse pass for fp32 inputs on the sm_103a tensor cores: 3xTF32.
//
// The Reverse procedure of "Exact tiled softmax attention with block-
// recomputed vector-Jacobian products" with frozen statistics,
//   p_ij = exp(s_ij - L_i),  gamma_ij = p_ij (G_i . V_j - delta_i),
//   dV_j += p_ij G_i,  dK_j += c gamma_ij Q_i   (tc_bwd32_kv_kernel, key-major)
//   dQ_i += c gamma_ij K_j                       (tc_bwd32_q_kernel, query-major)
// with delta_i = G_i . Y_i (HarshvardhanJ/FlashAttention, backward section),
// for fp32 inputs at close to fp32 accuracy, as the 3xTF32 forward does it:
// every product a b of the method is formed from three tf32 tensor-core
// products a_hi b_lo + a_lo b_hi + a_hi b_hi (x_hi = x rounded to tf32, x_lo =
// x - x_hi rounded to tf32), accumulated in fp32 in TMEM.  Each probability
// and gamma block is recomputed where it is needed; no n x n matrix is stored
// and dQ is written once per query block (no atomics).
//
// Widths d = v = 64.  A preparation kernel writes the tf32 parts of the
// operands that reach the tensor cores through shared memory: Q, dY, K, V
// row-major and Q^T, dY^T, K^T (so that every shared-memory operand is
// K-major).  The operand held for a whole CTA (K and V in the dK/dV kernel, Q
// and dY in the dQ kernel) is split by its own row's thread and kept in TMEM.
// delta_i and L_i log2(e) come from the delta kernel (padded vectors).
//
// tc_bwd32_kv_kernel -- one CTA = 128 keys of one slice; steps of 32 queries.
//   TMEM: K_hi, V_hi (64 columns each, A operands; K_lo, V_lo are A operands
//   in shared memory), dV, dK (64 each), and two buffers of S^T then P^T_hi,
//   P^T_lo, dP^T then dS^T_hi, dS^T_lo (32 each).  Per step: S^T = K Q^T,
//   dP^T = V dY^T; the elementwise warps (thread = key) form P^T and dS^T and
//   write their tf32 parts; dV += P^T dY, dK += dS^T Q.  S^T(t+1), dP^T(t+1)
//   run while the elementwise warps work on step t.  Every kPromote steps the
//   partial dV, dK rows go into the fp32 outputs.
// tc_bwd32_q_kernel -- one CTA = 128 queries of one slice; steps of 32 keys.
//   TMEM: Q_hi, Q_lo, dY_hi, dY_lo (64 each), dQ (64), and two buffers of
//   S then dS_hi, dP, dS_lo (32 each): S(t+1) and dP(t+1) run while the
//   elementwise warps (thread = query) form dS(t); dQ += dS K.
// Warps 0-3 elementwise (TMEM lane quarter = warp), warp 4 TMA, warp 5 MMA.
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
                   int box_rows);  // tc_fwd32.cu

namespace {

using namespace tc;

constexpr int kD = 64;        // d = v
constexpr int kBlk = 128;     // keys (dK/dV kernel) or queries (dQ kernel) per CTA
constexpr int kStep = 32;     // queries (dK/dV) or keys (dQ) per step
constexpr int kThreads = 192;
constexpr int kWarpTMA = 4;
constexpr int kWarpMMA = 5;
constexpr uint32_t kTmemCols = 512;
constexpr int kTile = kStep * kD * 4;  // one tf32 part of a 32 x 64 (or 64 x 32) tile: 8 KB
// The dK/dV kernel's TMEM accumulators restart every kPromote query steps:
// the fp32 accumulator of the tensor core loses low-order bits relative to its
// running sum in proportion to the number of steps (measured: normwise 5.7e-5
// on dK after 128 steps), so each partial sum of at most 1024 queries is added
// into the fp32 output row by its owning thread instead.
constexpr int kPromote = 32;

struct Bwd32Params {
  // dK/dV kernel, per query step: Q and dY (B of S^T, dP^T), Q^T and dY^T (B of dK, dV)
  CUtensorMap tqh, tql, tyh, tyl, tqth, tqtl, tyth, tytl;
  // dQ kernel, per key step: K and V (B of S, dP), K^T (B of dQ)
  CUtensorMap tkh, tkl, tvh, tvl, tkth, tktl;
  const float* Q;
  const float* K;
  const float* V;
  const float* dY;
  const float* delta;  // [BH][npad]
  const float* lse2;   // [BH][npad]: L log2(e), +inf on padding and empty rows
  float* dQ;
  float* dK;
  float* dV;
  int n, nk, off, npad, BH, mask_kind, window, words_per_row;
  const uint32_t* bits;
  float sl2;    // c log2(e)
  float scale;  // c
  unsigned* status;
};

// Allowed keys k0 .. k0+31 of query row i (bit e = key k0 + e).
__device__ __forceinline__ uint32_t range_bits32(int a, int b) {
  a = max(a, 0);
  b = min(b, 31);
  if (a > b) return 0u;
  const uint32_t width = static_cast<uint32_t>(b - a + 1);
  const uint32_t m = width == 32 ? 0xFFFFFFFFu : ((1u << width) - 1u);
  return m << a;
}
__device__ __forceinline__ uint32_t row_allow(const Bwd32Params& p, int i, int k0) {
  if (i >= p.n) return 0u;
  uint32_t a = range_bits32(0, p.nk - 1 - k0);
  const int ia = i + p.off;  // absolute position of row i
  if (p.mask_kind == kMaskCausal) a &= range_bits32(0, ia - k0);
  if (p.mask_kind == kMaskWindow) a &= range_bits32(ia - p.window + 1 - k0, ia - k0);
  if (p.mask_kind == kMaskBitmask) {
    const int w = k0 >> 5;
    a &= w < p.words_per_row ? __ldg(p.bits + static_cast<size_t>(i) * p.words_per_row + w) : 0u;
  }
  return a;
}
// Queries q0 .. q0+31 that may attend key j (bit e = query q0 + e).
__device__ __forceinline__ uint32_t col_allow(const Bwd32Params& p, int j, int q0) {
  if (j >= p.nk) return 0u;
  uint32_t a = range_bits32(0, p.n - 1 - q0);
  const int jq = j - p.off;  // the first query position that reaches key j
  if (p.mask_kind == kMaskCausal) a &= range_bits32(jq - q0, 31);
  if (p.mask_kind == kMaskWindow) a &= range_bits32(jq - q0, jq + p.window - 1 - q0);
  if (p.mask_kind == kMaskBitmask) {
    uint32_t b = 0u;
    const uint32_t* col = p.bits + (j >> 5);
#pragma unroll 4
    for (int e = 0; e < 32; ++e) {
      const int i = q0 + e;
      if (i < p.n) b |= ((__ldg(col + static_cast<size_t>(i) * p.words_per_row) >> (j & 31)) & 1u) << e;
    }
    a &= b;
  }
  return a;
}

// The tf32 hi / lo parts of a 64-wide fp32 row into TMEM (lane = the thread's
// row, columns [col, col + 64) for hi and [col + 64, col + 128) for lo); zeros
// for a row past the end.
__device__ __forceinline__ void row_to_tmem(const float* row, bool valid, uint32_t taddr) {
  const float4* r4 = reinterpret_cast<const float4*>(row);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t hi[32], lo[32];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float4 x = valid ? __ldg(r4 + 8 * c + e) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float h = tf32_hi(xs[u]);
        hi[4 * e + u] = __float_as_uint(h);
        lo[4 * e + u] = __float_as_uint(tf32_lo(xs[u], h));
      }
    }
    tmem_st32(taddr + 32 * c, hi);
    tmem_st32(taddr + 64 + 32 * c, lo);
  }
}

// fp32 values -> their tf32 hi parts (in place) and lo parts.
__device__ __forceinline__ void split32(uint32_t (&x)[32], uint32_t (&lo)[32]) {
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const float v = __uint_as_float(x[e]);
    const float h = tf32_hi(v);
    x[e] = __float_as_uint(h);
    lo[e] = __float_as_uint(tf32_lo(v, h));
  }
}

// The preparation kernel: tf32 hi / lo parts of Q, dY, K, V (tensor
// blockIdx.z = 0, 1, 2, 3), row-major like the input, and of Q, dY, K also
// transposed ([BH][64][ld], rows contiguous along the sequence).  One CTA per
// 32 rows of one slice.
__global__ void __launch_bounds__(256) split_bwd32_kernel(
    const float* Q, const float* dY, const float* K, const float* V, float* qh, float* ql,
    float* yh, float* yl, float* kh, float* kl, float* vh, float* vl, float* qth, float* qtl,
    float* yth, float* ytl, float* kth, float* ktl, int n, int nk, int ldq, int ldk) {
  __shared__ float tile[32][kD + 1];
  const int t = blockIdx.z, bh = blockIdx.y, r0 = blockIdx.x * 32;
  const int rows_all = t < 2 ? n : nk;
  if (r0 >= rows_all) return;
  const int rows = min(32, rows_all - r0);
  const float* src = t == 0 ? Q : t == 1 ? dY : t == 2 ? K : V;
  float* dh = t == 0 ? qh : t == 1 ? yh : t == 2 ? kh : vh;
  float* dl = t == 0 ? ql : t == 1 ? yl : t == 2 ? kl : vl;
  const size_t base = (static_cast<size_t>(bh) * rows_all + r0) * kD;
  for (int idx = threadIdx.x; idx < rows * kD; idx += 256) {
    const float x = __ldg(src + base + idx);
    const float h = tf32_hi(x);
    dh[base + idx] = h;
    dl[base + idx] = tf32_lo(x, h);
    tile[idx / kD][idx % kD] = x;
  }
  if (t == 3) return;
  __syncthreads();
  float* th = t == 0 ? qth : t == 1 ? yth : kth;
  float* tl = t == 0 ? qtl : t == 1 ? ytl : ktl;
  const int ld = t < 2 ? ldq : ldk;
  const size_t tbase = static_cast<size_t>(bh) * kD * ld + r0;
  for (int idx = threadIdx.x; idx < kD * 32; idx += 256) {
    const int c = idx >> 5, rr = idx & 31;
    if (rr < rows) {
      const float x = tile[rr][c];
      const float h = tf32_hi(x);
      th[tbase + static_cast<size_t>(c) * ld + rr] = h;
      tl[tbase + static_cast<size_t>(c) * ld + rr] = tf32_lo(x, h);
    }
  }
}

// Untiled bulk copy global -> shared (16-byte aligned, size a multiple of
// 16), completing on mbarrier `bar`.
__device__ __forceinline__ void bulk_load_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                    ~static_cast<uintptr_t>(1023));
}

// ===========================================================================
// Key-major kernel: dK, dV
// ===========================================================================
// Shared memory: NSS S halves (Q_lo, Q_hi, dY_lo, dY_hi: 32 queries x 64, in
// 128-byte-swizzled chunks of 32 rows x 32 columns, a chunk's lo and hi tiles
// adjacent), each free once S^T and dP^T of its step are done; NTS T halves (Q^T_hi, Q^T_lo, dY^T_hi, dY^T_lo:
// 64 rows x 32 queries, one chunk), each free once dK of its step is; NV
// slots of delta and L log2(e) for the step's 32 queries, free once the
// elementwise warps have read them; then K_lo and V_lo (128 keys x 64, the A
// operands of K_lo Q_hi^T and V_lo dY_hi^T), written by their rows' threads.
// TMEM: K_hi [0,64), V_hi [64,128), dV [128,192), dK [192,256) and two step
// buffers at 256 + 128 b of four 32-column blocks: S^T in two parts (then
// P^T_hi, P^T_lo), dP^T in two parts (then dS^T_hi, dS^T_lo).  The MMA warp
// issues S^T(t+1), dP^T(t+1) before dV(t), dK(t): the tensor pipe forms the
// next step's products while the elementwise warps form P^T(t), dS^T(t);
// dV(t) is issued once P^T(t) is written, dK(t) once dS^T(t) is.
// A tcgen05.mma of M = 128 costs about as much for N = 32 as for N = 64
// (measured: ~48 cycles each, 64 for N = 128), so S^T = K Q^T is formed as
// K_hi [Q_lo; Q_hi]^T (one N = 64 product: K_hi Q_lo^T into the first block,
// K_hi Q_hi^T into the second) plus K_lo Q_hi^T (N = 32, into the second
// block), and the elementwise threads add the two blocks: 16 instructions
// per product instead of 24.
struct KvLay32 {
  static constexpr int NSS = 3, NTS = 2, NV = 4;
  // S half: per 32-column chunk c the lo tile then the hi tile (4 KB each), so
  // that [Q_lo; Q_hi] of a chunk is one 64-row B operand
  static constexpr int QS = 0, YS = 2 * kTile, CHUNK = 2 * 4096, SHALF = 4 * kTile;
  static constexpr int QTH = 0, QTL = kTile, YTH = 2 * kTile, YTL = 3 * kTile, THALF = 4 * kTile;
  static constexpr int S_OFF = 0;
  static constexpr int T_OFF = S_OFF + NSS * SHALF;
  static constexpr int KLO_OFF = T_OFF + NTS * THALF;
  static constexpr int VLO_OFF = KLO_OFF + kBlk * kD * 4;
  static constexpr int VEC_OFF = VLO_OFF + kBlk * kD * 4;
  static constexpr int BAR_OFF = VEC_OFF + NV * 256;
  // B_A: K, V split; B_QSF / B_QSE, B_QTF / B_QTE, B_VF / B_VE: S half, T half,
  // vector slot full / free; B_SP: S^T, dP^T of a buffer done; B_P, B_DS: P^T,
  // dS^T parts of a buffer written; B_SEG: dV, dK of a kPromote-step segment
  // done; B_DONE: all products done; B_DRAIN: the MMA warp's last commit.
  static constexpr int B_A = 0, B_QSF = 1, B_QSE = B_QSF + NSS, B_QTF = B_QSE + NSS,
                       B_QTE = B_QTF + NTS, B_VF = B_QTE + NTS, B_VE = B_VF + NV,
                       B_SP = B_VE + NV, B_P = B_SP + 2, B_DS = B_P + 2, B_SEG = B_DS + 2,
                       B_DONE = B_SEG + 1, B_DRAIN = B_DONE + 1, NBAR = B_DRAIN + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;  // [0] TMEM base, [1] abort flag
  static constexpr int ALLOC = MISC_OFF + 16 + 1024;
  static constexpr uint32_t T_KH = 0, T_VH = 64, T_DV = 128, T_DK = 192, T_BUF = 256,
                            B_S = 0, B_PL = 32, B_DP = 64, B_DSL = 96, B_STRIDE = 128;
  static_assert(SHALF % 1024 == 0 && THALF % 1024 == 0, "1024-byte aligned tiles");
  static_assert(T_BUF + 2 * B_STRIDE <= kTmemCols, "TMEM columns");
  static_assert(ALLOC <= 232448, "shared memory");
};

// Row r of a 64-wide fp32 operand: its tf32 hi parts into TMEM (lane = r,
// columns [taddr, taddr + 64)) and its lo parts into row r of a K-major,
// 128-byte-swizzled shared-memory tile of 128 rows (two chunks of 32 columns,
// 16 KB apart); zeros for a row past the end.
__device__ __forceinline__ void row_split_tmem_smem(const float* row, bool valid, uint32_t taddr,
                                                    uint8_t* tile, int r) {
  const float4* r4 = reinterpret_cast<const float4*>(row);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t hi[32];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float4 x = valid ? __ldg(r4 + 8 * c + e) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float xs[4] = {x.x, x.y, x.z, x.w};
      float lo4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float h = tf32_hi(xs[u]);
        hi[4 * e + u] = __float_as_uint(h);
        lo4[u] = tf32_lo(xs[u], h);
      }
      *reinterpret_cast<float4*>(tile + c * (kBlk * 128) + r * 128 + ((e ^ (r & 7)) << 4)) =
          make_float4(lo4[0], lo4[1], lo4[2], lo4[3]);
    }
    tmem_st32(taddr + 32 * c, hi);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd32_kv_kernel(const __grid_constant__ Bwd32Params p) {
  using Lay = KvLay32;
  constexpr int NSS = Lay::NSS, NTS = Lay::NTS, NV = Lay::NV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + Lay::BAR_OFF;
  auto bar = [&](int k) { return bar0 + 8u * k; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  // Every role's waits are warp-uniform: a lane that timed out alone must not
  // leave the others in a warp-collective instruction.
  auto wait_warp = [&](int k, int parity) {
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar(k), static_cast<uint32_t>(parity), abort_flag));
  };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.n, nk = p.nk, off = p.off;
  const int bh = blockIdx.y;
  const int k0 = blockIdx.x * kBlk;  // low key blocks reach the most queries: first
  // Query steps that can reach keys k0 .. k1 (query i sits at position i + off).
  const int k1 = min(k0 + kBlk, nk) - 1;
  int q_begin = 0, q_end = n;
  if (p.mask_kind == kMaskCausal || p.mask_kind == kMaskWindow) q_begin = max(0, k0 - off);
  if (p.mask_kind == kMaskWindow) q_end = min(n, max(0, k1 - off + p.window));
  const int s_begin = q_begin / kStep;
  const int nsteps = q_end > q_begin ? (q_end + kStep - 1) / kStep - s_begin : 0;

  if (threadIdx.x == 0) {
    mbar_init(bar(Lay::B_A), kBlk);
    for (int s = 0; s < NSS; ++s) {
      mbar_init(bar(Lay::B_QSF + s), 1);
      mbar_init(bar(Lay::B_QSE + s), 1);
    }
    for (int s = 0; s < NTS; ++s) {
      mbar_init(bar(Lay::B_QTF + s), 1);
      mbar_init(bar(Lay::B_QTE + s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(bar(Lay::B_VF + s), 1);
      mbar_init(bar(Lay::B_VE + s), kBlk);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(Lay::B_SP + b), 1);
      mbar_init(bar(Lay::B_P + b), kBlk);
      mbar_init(bar(Lay::B_DS + b), kBlk);
    }
    mbar_init(bar(Lay::B_SEG), 1);
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
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp == kWarpTMA) {
    const bool leader = elect_one();
    if (leader) {
      prefetch_tmap(&p.tqh);
      prefetch_tmap(&p.tql);
      prefetch_tmap(&p.tyh);
      prefetch_tmap(&p.tyl);
      prefetch_tmap(&p.tqth);
      prefetch_tmap(&p.tqtl);
      prefetch_tmap(&p.tyth);
      prefetch_tmap(&p.tytl);
    }
    const uint64_t keep = policy_evict_last();  // read by every key block of the slice
    bool ok = true;
    int ns = 0, nt = 0, nv = 0;  // S halves, T halves, vector slots filled
    // The S half and the vectors of step s (issued one step ahead of the T half).
    auto load_s = [&](int s) {
      const int q0 = (s_begin + s) * kStep;
      const int slot = s % NSS, fill = s / NSS;
      if (fill >= 1 && !(ok = wait_warp(Lay::B_QSE + slot, (fill - 1) & 1)))
        return;
      const uint32_t sh = sbase + Lay::S_OFF + slot * Lay::SHALF, fs = bar(Lay::B_QSF + slot);
      if (leader) {
        mbar_arrive_expect_tx(fs, Lay::SHALF);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint32_t qc = sh + Lay::QS + c * Lay::CHUNK, yc = sh + Lay::YS + c * Lay::CHUNK;
          tma_load_3d(qc, &p.tql, fs, 32 * c, q0, bh, keep);
          tma_load_3d(qc + 4096, &p.tqh, fs, 32 * c, q0, bh, keep);
          tma_load_3d(yc, &p.tyl, fs, 32 * c, q0, bh, keep);
          tma_load_3d(yc + 4096, &p.tyh, fs, 32 * c, q0, bh, keep);
        }
      }
      ++ns;
      const int vs = s % NV, vfill = s / NV;
      if (vfill >= 1 && !(ok = wait_warp(Lay::B_VE + vs, (vfill - 1) & 1)))
        return;
      const uint32_t vec = sbase + Lay::VEC_OFF + vs * 256, fv = bar(Lay::B_VF + vs);
      if (leader) {
        mbar_arrive_expect_tx(fv, 256);
        const size_t vo = static_cast<size_t>(bh) * p.npad + q0;
        bulk_load_g2s(vec, p.delta + vo, 128, fv);
        bulk_load_g2s(vec + 128, p.lse2 + vo, 128, fv);
      }
      ++nv;
    };
    if (nsteps > 0) load_s(0);
    for (int it = 0; it < nsteps && ok; ++it) {
      if (it + 1 < nsteps) {
        load_s(it + 1);
        if (!ok) break;
      }
      const int slot = it % NTS, fill = it / NTS;
      if (fill >= 1 && !(ok = wait_warp(Lay::B_QTE + slot, (fill - 1) & 1)))
        break;
      const uint32_t th = sbase + Lay::T_OFF + slot * Lay::THALF, ft = bar(Lay::B_QTF + slot);
      const int q0 = (s_begin + it) * kStep;
      if (leader) {
        mbar_arrive_expect_tx(ft, Lay::THALF);
        tma_load_3d(th + Lay::QTH, &p.tqth, ft, q0, 0, bh, keep);
        tma_load_3d(th + Lay::QTL, &p.tqtl, ft, q0, 0, bh, keep);
        tma_load_3d(th + Lay::YTH, &p.tyth, ft, q0, 0, bh, keep);
        tma_load_3d(th + Lay::YTL, &p.tytl, ft, q0, 0, bh, keep);
      }
      ++nt;
    }
    __syncwarp();
    if (!ok && leader) {
      raise_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    // Never leave with copies in flight: the last fill of every slot.
    for (int u = 0; u < NSS && u < ns; ++u) {
      const int i = ns - 1 - u;
      mbar_wait_inflight(bar(Lay::B_QSF + i % NSS), (i / NSS) & 1);
    }
    for (int u = 0; u < NTS && u < nt; ++u) {
      const int i = nt - 1 - u;
      mbar_wait_inflight(bar(Lay::B_QTF + i % NTS), (i / NTS) & 1);
    }
    for (int u = 0; u < NV && u < nv; ++u) {
      const int i = nv - 1 - u;
      mbar_wait_inflight(bar(Lay::B_VF + i % NV), (i / NV) & 1);
    }
  } else if (warp == kWarpMMA) {
    // One elected lane runs the whole issue loop: it alone waits, issues and
    // commits; the other lanes wait for it at the end.
    const bool leader = elect_one();
    constexpr uint32_t kIdS = idesc_tf32(kBlk, kStep), kIdS2 = idesc_tf32(kBlk, 2 * kStep);
    constexpr uint32_t kIdAcc = idesc_tf32(kBlk, kD);
    // One descriptor base for every shared-memory operand (tiles 1024-byte
    // aligned, 8-row groups 1024 bytes apart); an operand adds its offset in
    // units of 16 bytes.
    const uint64_t d0 = sdesc_sw128(sbase, 16, 1024);
    // S^T = K Q^T or dP^T = V dY^T of step t into buffer t & 1, over 8 K-steps
    // of the width: A_hi [B_lo; B_hi]^T (N = 64, A_hi in TMEM, B the chunk's lo
    // and hi tiles of the S half) into blocks 0 and 1, then A_lo B_hi^T (N = 32,
    // A_lo in shared memory: 128 rows, chunks 16 KB apart) into block 1.
    auto issue_xt = [&](uint32_t d, uint32_t a_hi, uint32_t a_lo, uint64_t b) {
#pragma unroll
      for (int kk = 0; kk < kD / 8; ++kk)
        mma_ts_tf32(d, a_hi + 8 * kk, b + (((kk >> 2) * Lay::CHUNK + (kk & 3) * 32) >> 4), kIdS2,
                    kk > 0 ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < kD / 8; ++kk)
        mma_ss_tf32(d + kStep, d0 + ((a_lo + (kk >> 2) * (kBlk * 128) + (kk & 3) * 32) >> 4),
                    b + (((kk >> 2) * Lay::CHUNK + 4096 + (kk & 3) * 32) >> 4), kIdS, 1u);
    };
    auto issue_step = [&](int t) {
      const uint64_t sd = d0 + ((Lay::S_OFF + (t % NSS) * Lay::SHALF) >> 4);
      const uint32_t buf = tmem + Lay::T_BUF + Lay::B_STRIDE * (t & 1);
      issue_xt(buf + Lay::B_S, tmem + Lay::T_KH, Lay::KLO_OFF, sd + (Lay::QS >> 4));
      issue_xt(buf + Lay::B_DP, tmem + Lay::T_VH, Lay::VLO_OFF, sd + (Lay::YS >> 4));
    };
    // D[128 x 64] += A[128 x 32] B^T over 4 K-steps (the step's queries), three
    // products; A = the hi / lo parts in the step's TMEM buffer, B = a 64 x 32
    // tile of the T half.
    auto issue_acc = [&](uint32_t d, uint32_t a_hi, uint32_t a_lo, uint64_t b_hi, uint64_t b_lo,
                         bool first) {
#pragma unroll
      for (int part = 0; part < 3; ++part) {
        const uint32_t a = part == 1 ? a_lo : a_hi;
        const uint64_t b = part == 0 ? b_lo : b_hi;
#pragma unroll
        for (int kk = 0; kk < kStep / 8; ++kk)
          mma_ts_tf32(d, a + 8 * kk, b + ((kk * 32) >> 4), kIdAcc,
                      (first && part == 0 && kk == 0) ? 0u : 1u);
      }
    };
    bool ok = true;
    if (leader) {
      ok = mbar_wait(bar(Lay::B_A), 0, abort_flag);
      tc_fence_after();
      // S^T(0), dP^T(0); then per step t: S^T(t+1), dP^T(t+1), dV(t), dK(t).
      // S^T(t+2) overwrites buffer t & 1 after dV(t), dK(t) have read it (the
      // tensor pipe runs one thread's MMAs in issue order), and the elementwise
      // warps write P^T(t+2) there only after S^T(t+2) is done.
      if (ok && nsteps > 0 && (ok = mbar_wait(bar(Lay::B_QSF), 0, abort_flag))) {
        tc_fence_after();
        issue_step(0);
        tc_commit(bar(Lay::B_SP));
        tc_commit(bar(Lay::B_QSE));
      }
      for (int it = 0; it < nsteps && ok; ++it) {
        const int b = it & 1;
        if (it + 1 < nsteps) {
          const int s1 = (it + 1) % NSS;
          if (!(ok = mbar_wait(bar(Lay::B_QSF + s1), ((it + 1) / NSS) & 1, abort_flag))) break;
          tc_fence_after();
          issue_step(it + 1);
          tc_commit(bar(Lay::B_SP + ((it + 1) & 1)));
          tc_commit(bar(Lay::B_QSE + s1));
        }
        const int ts = it % NTS;
        const uint64_t td = d0 + ((Lay::T_OFF + ts * Lay::THALF) >> 4);
        const uint32_t buf = tmem + Lay::T_BUF + Lay::B_STRIDE * b;
        // The accumulators restart at every kPromote-th step: the elementwise
        // warps have moved the partial sums out before writing P^T(it).
        const bool first = it % kPromote == 0;
        if (!(ok = mbar_wait(bar(Lay::B_QTF + ts), (it / NTS) & 1, abort_flag))) break;
        if (!(ok = mbar_wait(bar(Lay::B_P + b), (it >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        // dV += P^T dY
        issue_acc(tmem + Lay::T_DV, buf + Lay::B_S, buf + Lay::B_PL, td + (Lay::YTH >> 4),
                  td + (Lay::YTL >> 4), first);
        if (!(ok = mbar_wait(bar(Lay::B_DS + b), (it >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        // dK += dS^T Q (c applied when the rows leave TMEM)
        issue_acc(tmem + Lay::T_DK, buf + Lay::B_DP, buf + Lay::B_DSL, td + (Lay::QTH >> 4),
                  td + (Lay::QTL >> 4), first);
        if ((it + 1) % kPromote == 0 && it + 1 < nsteps) tc_commit(bar(Lay::B_SEG));
        tc_commit(bar(Lay::B_QTE + ts));
      }
      tc_commit(bar(Lay::B_DONE));
      if (!ok) {
        raise_status(p.status, kStatusTimeout);
        *abort_flag = 1;
      }
      // Every MMA issued has completed before TMEM is freed, abort or not.
      tc_commit(bar(Lay::B_DRAIN));
    }
    __syncwarp();
    mbar_wait_inflight(bar(Lay::B_DRAIN), 0);
  } else {
    // Elementwise: thread = key j = k0 + r (TMEM lane r); its 32 columns of a
    // step are the step's queries.
    const int r = warp * 32 + lane;
    const int j = k0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const size_t jrow = (static_cast<size_t>(bh) * nk + (j < nk ? j : 0)) * kD;
    row_split_tmem_smem(p.K + jrow, j < nk, tmem + lane_off + Lay::T_KH, smem + Lay::KLO_OFF, r);
    row_split_tmem_smem(p.V + jrow, j < nk, tmem + lane_off + Lay::T_VH, smem + Lay::VLO_OFF, r);
    tmem_st_wait();
    fence_proxy_async_smem();  // the lo tiles are read by the tensor core
    tc_fence_before();
    mbar_arrive(bar(Lay::B_A));
    const float sl2 = p.sl2;
    bool ok = true;
    // The partial dV_j, c dK_j in TMEM into the fp32 output rows: stored by
    // the first move, added by the later ones (this thread alone writes row j,
    // in program order, so the sum is deterministic).
    auto move_out = [&](bool first_move) {
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        float* dst = (which == 0 ? p.dV : p.dK) + jrow;
        const float mul = which == 0 ? 1.f : p.scale;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + (which == 0 ? Lay::T_DV : Lay::T_DK) + 32 * c, o);
          tmem_ld_wait();
          reg_fence(o);
          if (j < nk) {
            float4* d4 = reinterpret_cast<float4*>(dst + 32 * c);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float4 v4 =
                  make_float4(__uint_as_float(o[4 * e]) * mul, __uint_as_float(o[4 * e + 1]) * mul,
                              __uint_as_float(o[4 * e + 2]) * mul,
                              __uint_as_float(o[4 * e + 3]) * mul);
              if (first_move)
                d4[e] = v4;
              else
                red_add_v4(reinterpret_cast<float*>(d4 + e), v4.x, v4.y, v4.z, v4.w);
            }
          }
        }
      }
    };
    for (int it = 0; it < nsteps; ++it) {
      const int q0 = (s_begin + it) * kStep;
      const int b = it & 1, vs = it % NV;
      const uint32_t tb = tmem + lane_off + Lay::T_BUF + Lay::B_STRIDE * b;
      const uint32_t allow = col_allow(p, j, q0);  // needs no product: before the waits
      if (!(ok = wait_warp(Lay::B_VF + vs, (it / NV) & 1))) break;
      if (!(ok = wait_warp(Lay::B_SP + b, (it >> 1) & 1))) break;
      tc_fence_after();
      if (it > 0 && it % kPromote == 0) {
        // dV, dK of the last kPromote steps are done: move them out before
        // dV(it), dK(it) restart the accumulators.
        if (!(ok = wait_warp(Lay::B_SEG, (it / kPromote - 1) & 1))) break;
        tc_fence_after();
        move_out(it == kPromote);
      }
      const float* dvec = reinterpret_cast<const float*>(smem + Lay::VEC_OFF + vs * 256);
      const float* lvec = dvec + 32;
      uint32_t s[32], dp[32], lo[32], t2[32];
      tmem_ld32(tb + Lay::B_S, s);
      tmem_ld32(tb + Lay::B_S + kStep, lo);
      tmem_ld32(tb + Lay::B_DP, dp);
      tmem_ld32(tb + Lay::B_DP + kStep, t2);
      tmem_ld_wait();
      reg_fence(s);
      reg_fence(lo);
      reg_fence(dp);
      reg_fence(t2);
#pragma unroll
      for (int e = 0; e < 32; ++e) {  // the two parts of S^T and of dP^T
        s[e] = __float_as_uint(__uint_as_float(s[e]) + __uint_as_float(lo[e]));
        dp[e] = __float_as_uint(__uint_as_float(dp[e]) + __uint_as_float(t2[e]));
      }
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(lvec + e);
        const float4 d4 = *reinterpret_cast<const float4*>(dvec + e);
        const float la[4] = {l4.x, l4.y, l4.z, l4.w}, da[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float pij =
              ((allow >> (e + u)) & 1u) ? ex2(fmaf(__uint_as_float(s[e + u]), sl2, -la[u])) : 0.f;
          s[e + u] = __float_as_uint(pij);
          dp[e + u] = __float_as_uint(pij * (__uint_as_float(dp[e + u]) - da[u]));
        }
      }
      mbar_arrive(bar(Lay::B_VE + vs));  // the vectors are in registers
      split32(s, lo);
      tmem_st32(tb + Lay::B_S, s);
      tmem_st32(tb + Lay::B_PL, lo);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Lay::B_P + b));
      split32(dp, lo);
      tmem_st32(tb + Lay::B_DP, dp);
      tmem_st32(tb + Lay::B_DSL, lo);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Lay::B_DS + b));
    }
    // Epilogue: the last partial dV_j, c dK_j (zeros when no query reaches the
    // block).  The TMEM reads are warp-collective: ok and the wait are uniform.
    const bool have = ok && nsteps > 0 && wait_warp(Lay::B_DONE, 0);
    if (ok && nsteps > 0 && !have) ok = false;
    tc_fence_after();
    if (have) {
      move_out(nsteps <= kPromote);
    } else if (j < nk) {
      float4* dv4 = reinterpret_cast<float4*>(p.dV + jrow);
      float4* dk4 = reinterpret_cast<float4*>(p.dK + jrow);
#pragma unroll 4
      for (int e = 0; e < kD / 4; ++e) dv4[e] = dk4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
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

// ===========================================================================
// Query-major kernel: dQ
// ===========================================================================
// Shared memory: NST stages of six 8 KB tiles -- K_hi, K_lo, V_hi, V_lo (32
// keys x 64, two chunks of 32 rows x 32 columns) and K^T_hi, K^T_lo (64 rows x
// 32 keys, one chunk).
struct QLay32 {
  static constexpr int NST = 4;
  static constexpr int KH = 0, KL = kTile, VH = 2 * kTile, VL = 3 * kTile, KTH = 4 * kTile,
                       KTL = 5 * kTile, STAGE = 6 * kTile;
  static constexpr int BAR_OFF = NST * STAGE;
  // B_A: Q, dY in TMEM; B_KF / B_KE: stage full / free; B_SP: S, dP of a
  // buffer done; B_DS: dS parts of a buffer written; B_DONE: dQ done.
  static constexpr int B_A = 0, B_KF = 1, B_KE = B_KF + NST, B_SP = B_KE + NST, B_DS = B_SP + 2,
                       B_DONE = B_DS + 2, B_DRAIN = B_DONE + 1, NBAR = B_DRAIN + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int ALLOC = MISC_OFF + 16 + 1024;
  // TMEM columns (Q_lo, dY_lo 64 after Q_hi, dY_hi); buffer b at 96 b.
  static constexpr uint32_t T_QH = 0, T_YH = 128, T_DQ = 256, T_S = 320, T_DP = 352, T_DSL = 384,
                            T_BUF = 96;
  static_assert(T_DSL + T_BUF + kStep <= kTmemCols, "TMEM columns");
  static_assert(ALLOC <= 232448, "shared memory");
};

__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd32_q_kernel(const __grid_constant__ Bwd32Params p) {
  using Lay = QLay32;
  constexpr int NST = Lay::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + Lay::BAR_OFF;
  auto bar = [&](int k) { return bar0 + 8u * k; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.n, nk = p.nk, off = p.off;
  const int bh = blockIdx.y;
  const int nqb = (n + kBlk - 1) / kBlk;
  const int q0 = (nqb - 1 - blockIdx.x) * kBlk;  // heaviest (causal) query blocks first
  const int q1 = min(q0 + kBlk, n) - 1;
  // Key steps that rows q0 .. q1 (at positions q0 + off ..) can reach.
  int k_begin = 0, k_end = nk;
  if (p.mask_kind == kMaskCausal || p.mask_kind == kMaskWindow) k_end = max(0, min(nk, q1 + off + 1));
  if (p.mask_kind == kMaskWindow) k_begin = min(k_end, max(0, q0 + off - p.window + 1));
  const int s_begin = k_begin / kStep;
  const int nsteps = k_end > k_begin ? (k_end + kStep - 1) / kStep - s_begin : 0;

  if (threadIdx.x == 0) {
    mbar_init(bar(Lay::B_A), kBlk);
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar(Lay::B_KF + s), 1);
      mbar_init(bar(Lay::B_KE + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(Lay::B_SP + b), 1);
      mbar_init(bar(Lay::B_DS + b), kBlk);
    }
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
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp == kWarpTMA) {
    const bool leader = elect_one();
    if (leader) {
      prefetch_tmap(&p.tkh);
      prefetch_tmap(&p.tkl);
      prefetch_tmap(&p.tvh);
      prefetch_tmap(&p.tvl);
      prefetch_tmap(&p.tkth);
      prefetch_tmap(&p.tktl);
    }
    const uint64_t keep = policy_evict_last();  // read by every query block of the slice
    bool ok = true;
    int fills = 0;
    for (int it = 0; it < nsteps && ok; ++it) {
      const int slot = it % NST, fill = it / NST;
      if (fill >= 1 && !(ok = mbar_wait(bar(Lay::B_KE + slot), (fill - 1) & 1, abort_flag))) break;
      const uint32_t st = sbase + slot * Lay::STAGE, fb = bar(Lay::B_KF + slot);
      const int k0 = (s_begin + it) * kStep;
      if (leader) {
        mbar_arrive_expect_tx(fb, Lay::STAGE);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          tma_load_3d(st + Lay::KH + c * 4096, &p.tkh, fb, 32 * c, k0, bh, keep);
          tma_load_3d(st + Lay::KL + c * 4096, &p.tkl, fb, 32 * c, k0, bh, keep);
          tma_load_3d(st + Lay::VH + c * 4096, &p.tvh, fb, 32 * c, k0, bh, keep);
          tma_load_3d(st + Lay::VL + c * 4096, &p.tvl, fb, 32 * c, k0, bh, keep);
        }
        tma_load_3d(st + Lay::KTH, &p.tkth, fb, k0, 0, bh, keep);
        tma_load_3d(st + Lay::KTL, &p.tktl, fb, k0, 0, bh, keep);
      }
      ++fills;
    }
    __syncwarp();
    if (!ok && leader) {
      raise_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    // Never leave with copies in flight: the last fill of every stage.
    for (int u = 0; u < NST && u < fills; ++u) {
      const int i = fills - 1 - u;
      mbar_wait_inflight(bar(Lay::B_KF + i % NST), (i / NST) & 1);
    }
  } else if (warp == kWarpMMA) {
    const bool leader = elect_one();
    constexpr uint32_t kIdS = idesc_tf32(kBlk, kStep);
    constexpr uint32_t kIdQ = idesc_tf32(kBlk, kD);
    const uint64_t d0 = sdesc_sw128(sbase, 16, 1024);
    bool ok = mbar_wait(bar(Lay::B_A), 0, abort_flag);
    tc_fence_after();
    // S(t) = Q K_t^T and dP(t) = dY V_t^T into buffer t % 2: three tf32
    // products each over 8 K-steps (A in TMEM, B = 32 x 64 stage tile).
    auto issue_sdp = [&](int t) {
      const int slot = t % NST, b = t & 1;
      const uint32_t st = slot * Lay::STAGE;
      if (leader) {
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const uint32_t dcol = (which == 0 ? Lay::T_S : Lay::T_DP) + Lay::T_BUF * b;
          const uint32_t acol = which == 0 ? Lay::T_QH : Lay::T_YH;
          const int bh_ = which == 0 ? Lay::KH : Lay::VH, bl_ = which == 0 ? Lay::KL : Lay::VL;
#pragma unroll
          for (int part = 0; part < 3; ++part) {
            const uint32_t a = tmem + acol + (part == 1 ? 64u : 0u);
            const uint64_t bd = d0 + ((st + (part == 0 ? bl_ : bh_)) >> 4);
#pragma unroll
            for (int kk = 0; kk < kD / 8; ++kk) {
              const uint32_t o16 = ((kk >> 2) * 4096 + (kk & 3) * 32) >> 4;
              mma_ts_tf32(tmem + dcol, a + 8 * kk, bd + o16, kIdS, (part > 0 || kk > 0) ? 1u : 0u);
            }
          }
        }
        tc_commit(bar(Lay::B_SP + b));
      }
    };
    auto k_full = [&](int t) {
      return mbar_wait(bar(Lay::B_KF + t % NST), (t / NST) & 1, abort_flag);
    };
    if (nsteps > 0 && ok && (ok = k_full(0))) {
      tc_fence_after();
      issue_sdp(0);
    }
    for (int t = 0; t < nsteps && ok; ++t) {
      // S(t+1), dP(t+1) into the other buffer: they run while the elementwise
      // warps form dS(t).  Its dS(t-1) was read by dQ(t-1), issued earlier.
      if (t + 1 < nsteps) {
        if (!(ok = k_full(t + 1))) break;
        tc_fence_after();
        issue_sdp(t + 1);
      }
      const int b = t & 1;
      if (!(ok = mbar_wait(bar(Lay::B_DS + b), (t >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      // dQ += dS(t) K_t: A = dS parts (TMEM, 4 K-steps over the step's keys),
      // B = K_t^T (64 x 32 stage tile).
      const uint32_t st = (t % NST) * Lay::STAGE;
      if (leader) {
#pragma unroll
        for (int part = 0; part < 3; ++part) {
          const uint32_t a = tmem + (part == 1 ? Lay::T_DSL : Lay::T_S) + Lay::T_BUF * b;
          const uint64_t bd = d0 + ((st + (part == 0 ? Lay::KTL : Lay::KTH)) >> 4);
#pragma unroll
          for (int kk = 0; kk < kStep / 8; ++kk)
            mma_ts_tf32(tmem + Lay::T_DQ, a + 8 * kk, bd + ((kk * 32) >> 4), kIdQ,
                        (t == 0 && part == 0 && kk == 0) ? 0u : 1u);
        }
        tc_commit(bar(Lay::B_KE + t % NST));
      }
    }
    if (leader) tc_commit(bar(Lay::B_DONE));
    __syncwarp();
    if (!ok && leader) {
      raise_status(p.status, kStatusTimeout);
      *abort_flag = 1;
    }
    if (leader) tc_commit(bar(Lay::B_DRAIN));
    mbar_wait_inflight(bar(Lay::B_DRAIN), 0);
  } else {
    // Elementwise: thread = query row i = q0 + r (TMEM lane r); its 32 columns
    // of a step are the step's keys.
    const int r = warp * 32 + lane;
    const int i = q0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const size_t irow = (static_cast<size_t>(bh) * n + (i < n ? i : 0)) * kD;
    row_to_tmem(p.Q + irow, i < n, tmem + lane_off + Lay::T_QH);
    row_to_tmem(p.dY + irow, i < n, tmem + lane_off + Lay::T_YH);
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(bar(Lay::B_A));
    const size_t vo = static_cast<size_t>(bh) * p.npad + q0 + r;  // q0 + r < npad
    const float dl = __ldg(p.delta + vo), lse2 = __ldg(p.lse2 + vo);
    const float sl2 = p.sl2;
    bool ok = true;
    for (int t = 0; t < nsteps; ++t) {
      const int b = t & 1;
      const uint32_t allow = row_allow(p, i, (s_begin + t) * kStep);  // before the wait
      if (!(ok = mbar_wait(bar(Lay::B_SP + b), (t >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      uint32_t s[32], dp[32], lo[32];
      tmem_ld32(tmem + lane_off + Lay::T_S + Lay::T_BUF * b, s);
      tmem_ld32(tmem + lane_off + Lay::T_DP + Lay::T_BUF * b, dp);
      tmem_ld_wait();
      reg_fence(s);
      reg_fence(dp);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float pij =
            ((allow >> e) & 1u) ? ex2(fmaf(__uint_as_float(s[e]), sl2, -lse2)) : 0.f;
        s[e] = __float_as_uint(pij * (__uint_as_float(dp[e]) - dl));  // dS
      }
      split32(s, lo);
      tmem_st32(tmem + lane_off + Lay::T_S + Lay::T_BUF * b, s);
      tmem_st32(tmem + lane_off + Lay::T_DSL + Lay::T_BUF * b, lo);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Lay::B_DS + b));
    }
    // Epilogue: c dQ_i, an fp32 row (zeros when the block reaches no key).  The
    // TMEM reads are warp-collective: the predicate is the warp's.
    const bool have = __all_sync(
        0xFFFFFFFFu, ok && nsteps > 0 && mbar_wait(bar(Lay::B_DONE), 0, abort_flag));
    if (ok && nsteps > 0 && !have) ok = false;
    tc_fence_after();
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      uint32_t o[32];
      if (have) {
        tmem_ld32(tmem + lane_off + Lay::T_DQ + 32 * c, o);
        tmem_ld_wait();
        reg_fence(o);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
      if (i < n) {
        float4* d4 = reinterpret_cast<float4*>(p.dQ + irow + 32 * c);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          d4[e] = make_float4(__uint_as_float(o[4 * e]) * p.scale,
                              __uint_as_float(o[4 * e + 1]) * p.scale,
                              __uint_as_float(o[4 * e + 2]) * p.scale,
                              __uint_as_float(o[4 * e + 3]) * p.scale);
      }
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

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace

// Workspace of the 3xTF32 reverse pass (after the reverse pass's own parts):
// the tf32 hi / lo parts of Q, dY, K, V row-major and of Q, dY, K transposed
// (rows padded to a multiple of 32 elements).
Bwd32Split bwd32_layout(const Problem& p, void* base) {
  const size_t ldq = (static_cast<size_t>(p.n) + 31) / 32 * 32;
  const size_t ldk = (static_cast<size_t>(p.nk) + 31) / 32 * 32;
  const size_t bq = align256(4 * static_cast<size_t>(p.BH) * p.n * kD);
  const size_t bk = align256(4 * static_cast<size_t>(p.BH) * p.nk * kD);
  const size_t btq = align256(4 * static_cast<size_t>(p.BH) * kD * ldq);
  const size_t btk = align256(4 * static_cast<size_t>(p.BH) * kD * ldk);
  const uintptr_t b = reinterpret_cast<uintptr_t>(base);
  Bwd32Split w;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    float* f = reinterpret_cast<float*>(b + o);
    o += bytes;
    return f;
  };
  w.qh = take(bq);
  w.ql = take(bq);
  w.yh = take(bq);
  w.yl = take(bq);
  w.kh = take(bk);
  w.kl = take(bk);
  w.vh = take(bk);
  w.vl = take(bk);
  w.qth = take(btq);
  w.qtl = take(btq);
  w.yth = take(btq);
  w.ytl = take(btq);
  w.kth = take(btk);
  w.ktl = take(btk);
  w.ldq = static_cast<int>(ldq);
  w.ldk = static_cast<int>(ldk);
  w.bytes = o;
  return w;
}

size_t bwd32_bytes(const Problem& p) { return bwd32_layout(p, nullptr).bytes; }

bool tc_bwd32_supported(const Problem& p) {
  if (p.dtype != kF32 || p.d != kD || p.v != kD || p.drop_t != 0) return false;
  return tmap_encoder() != nullptr;
}

cudaError_t launch_tc_bwd32(const BwdArgs& a, const Bwd32Split& w, cudaStream_t s) {
  const Problem& pr = a.p;
  Bwd32Params p;
  const int BH = pr.BH, n = pr.n, nk = pr.nk;
  if (!make_tmap_f32(&p.tqh, w.qh, kD, kD, n, BH, kStep) ||
      !make_tmap_f32(&p.tql, w.ql, kD, kD, n, BH, kStep) ||
      !make_tmap_f32(&p.tyh, w.yh, kD, kD, n, BH, kStep) ||
      !make_tmap_f32(&p.tyl, w.yl, kD, kD, n, BH, kStep) ||
      !make_tmap_f32(&p.tqth, w.qth, n, w.ldq, kD, BH, kD) ||
      !make_tmap_f32(&p.tqtl, w.qtl, n, w.ldq, kD, BH, kD) ||
      !make_tmap_f32(&p.tyth, w.yth, n, w.ldq, kD, BH, kD) ||
      !make_tmap_f32(&p.tytl, w.ytl, n, w.ldq, kD, BH, kD) ||
      !make_tmap_f32(&p.tkh, w.kh, kD, kD, nk, BH, kStep) ||
      !make_tmap_f32(&p.tkl, w.kl, kD, kD, nk, BH, kStep) ||
      !make_tmap_f32(&p.tvh, w.vh, kD, kD, nk, BH, kStep) ||
      !make_tmap_f32(&p.tvl, w.vl, kD, kD, nk, BH, kStep) ||
      !make_tmap_f32(&p.tkth, w.kth, nk, w.ldk, kD, BH, kD) ||
      !make_tmap_f32(&p.tktl, w.ktl, nk, w.ldk, kD, BH, kD))
    return cudaErrorInvalidValue;
  p.Q = static_cast<const float*>(a.Q);
  p.K = static_cast<const float*>(a.K);
  p.V = static_cast<const float*>(a.V);
  p.dY = static_cast<const float*>(a.dY);
  p.delta = a.delta;
  p.lse2 = a.lse2;
  p.dQ = static_cast<float*>(a.dQ);
  p.dK = static_cast<float*>(a.dK);
  p.dV = static_cast<float*>(a.dV);
  p.n = n;
  p.nk = nk;
  p.off = nk - n;
  p.npad = a.npad;
  p.BH = BH;
  p.mask_kind = pr.mask_kind;
  p.window = pr.window;
  p.words_per_row = pr.words_per_row;
  p.bits = pr.bitmask;
  p.sl2 = pr.scale * kLog2e;
  p.scale = pr.scale;
  p.status = a.status;
  cudaError_t e =
      cudaFuncSetAttribute(tc_bwd32_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           KvLay32::ALLOC);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_bwd32_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             QLay32::ALLOC);
  if (e != cudaSuccess) {
    record_error("tc_bwd32: cudaFuncSetAttribute", static_cast<int>(e), cudaGetErrorString(e));
    return e;
  }
  const int rows = n > nk ? n : nk;
  before_launch(kKernSplit32, s);
  split_bwd32_kernel<<<dim3((rows + 31) / 32, BH, 4), 256, 0, s>>>(
      p.Q, p.dY, p.K, p.V, w.qh, w.ql, w.yh, w.yl, w.kh, w.kl, w.vh, w.vl, w.qth, w.qtl, w.yth,
      w.ytl, w.kth, w.ktl, n, nk, w.ldq, w.ldk);
  after_launch(kKernSplit32, s);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  before_launch(kKernBwd, s);
  before_launch(kKernBwdQ, s);
  tc_bwd32_q_kernel<<<dim3((n + kBlk - 1) / kBlk, BH), kThreads, QLay32::ALLOC, s>>>(p);
  e = cudaGetLastError();
  after_launch(kKernBwdQ, s);
  if (e == cudaSuccess) {
    tc_bwd32_kv_kernel<<<dim3((nk + kBlk - 1) / kBlk, BH), kThreads, KvLay32::ALLOC, s>>>(p);
    e = cudaGetLastError();
  }
  after_launch(kKernBwd, s);
  return e;
}

}  // namespace exattn
