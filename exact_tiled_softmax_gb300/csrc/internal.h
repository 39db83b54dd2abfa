// Internal (host + device) declarations of libexattn: problem description and
// the kernel launchers behind the C ABI in include/exattn.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace exattn {

enum { kMaskNone = 0, kMaskCausal = 1, kMaskWindow = 2, kMaskBitmask = 3 };
enum { kF32 = 0, kBF16 = 1 };

// The workspace of every entry point starts with a 256-byte area that the
// host clears before the first launch: word 0 is the status word; words
// kSchedWord and kSchedWord + 1 count the items that the persistent kernels
// of one call (forward; or dK/dV, then dQ) have handed out.
constexpr size_t kStatusBytes = 256;
constexpr int kSchedWord = 16;

// One attention problem: BH = batch*heads independent slices; n query rows
// against nk keys (nk == n for self-attention shapes).  Query i sits at
// absolute position i + nk - n: the causal and window masks compare keys with
// that position, and bit rows are [n][ceil(nk/32)].
struct Problem {
  int BH, n, d, v, dtype;
  int nk;
  float scale;
  int mask_kind, window, words_per_row;
  const uint32_t* bitmask;
  // Dropout (drop_t == 0: none): key j of row i in slice bh is kept when the
  // 16-bit Philox value u_ij >= drop_t; kept entries are scaled by drop_scale.
  uint32_t drop_t;
  float drop_scale;
  uint32_t seed_lo, seed_hi;
};

struct FwdArgs {
  Problem p;
  const void* Q;
  const void* K;
  const void* V;
  void* Y;
  float* L;
  unsigned* status;
};

struct BwdArgs {
  Problem p;
  const void* Q;
  const void* K;
  const void* V;
  const void* Y;
  const void* dY;
  const float* L;
  void* dQ;
  void* dK;
  void* dV;
  int npad;       // n rounded up to a multiple of 128
  float* delta;   // [BH][npad] workspace: delta_i (0 on padding rows)
  float* lse2;    // [BH][npad] workspace: L_i * log2(e); +inf on padding / empty rows
  float* dQacc;   // [BH][n][d] fp32 workspace, zeroed by the launcher
  unsigned* status;
};

// Profiling hooks (api.cu): every kernel launch goes through these so the
// launch counter and the one-shot event hooks see it.
enum KernelRole {
  kKernFwd = 0,
  kKernDelta = 1,
  kKernBwd = 2,
  kKernDqConvert = 3,
  kKernBwdQ = 4,
  kKernSplitPartial = 5,
  kKernSplitMerge = 6,
  kKernSplit32 = 7,
  kKernRoles = 8
};
void before_launch(int role, cudaStream_t s);
// Remember the last failing step of this host thread (exattn_last_error).
void record_error(const char* where, int code, const char* detail);
void after_launch(int role, cudaStream_t s);

// SIMT fp32 kernels (any dtype, d, v <= 256).  launch_simt_bwd uses the
// register-tiled reverse kernel for d, v in {64, 128} and the general one
// otherwise.
cudaError_t launch_simt_fwd(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_simt_bwd(const BwdArgs& a, cudaStream_t s);
bool simt_bwd_rt_supported(const Problem& p);
cudaError_t launch_simt_bwd_rt(const BwdArgs& a, cudaStream_t s);

// delta_i = dY_i . Y_i and the log2-scaled row statistic (memory-bound
// preprocessing of the reverse pass), written to padded [BH][npad] vectors.
cudaError_t launch_delta(const BwdArgs& a, cudaStream_t s);
// dQ = dQacc converted to the output dtype.
cudaError_t launch_dq_convert(const BwdArgs& a, cudaStream_t s);

// tcgen05 / TMA / TMEM kernels (bf16, d = v in {64, 128}).
// The reverse pass has two forms: the split form (a key-major dK/dV kernel and
// a query-major dQ kernel, no atomics; the default) and the atomic form (one
// key-major kernel adding dQ into an fp32 accumulator).
bool tc_bwd_split_supported(const Problem& p);
cudaError_t launch_tc_bwd_split(const BwdArgs& a, cudaStream_t s);
bool tc_fwd_supported(const Problem& p);
cudaError_t launch_tc_fwd(const FwdArgs& a, cudaStream_t s);
// The same kernel in split-KV summary mode: chunks of chunk_keys (a multiple
// of 128) keys, summaries to pm / pl / pz [BH][splits][n] (see SplitArgs).
cudaError_t launch_tc_fwd_chunks(const FwdArgs& a, int chunk_keys, int splits, float* pm,
                                 float* pl, float* pz, cudaStream_t s);
bool tc_bwd_supported(const Problem& p);
cudaError_t launch_tc_bwd(const BwdArgs& a, cudaStream_t s);

// 3xTF32 tensor-core forward for fp32 inputs (d = v in {64, 128}).  K and V
// are first split into tf32 hi / lo parts (V transposed) in the workspace.
struct Split32 {
  float* kh;   // [BH][nk][d]
  float* kl;
  float* vth;  // [BH][v][ldt], keys contiguous
  float* vtl;
  int ldt;     // nk rounded up to 32
};
bool tc_fwd32_shape(int d, int v);  // widths the 3xTF32 forward takes (fp32)
bool tc_fwd32_supported(const Problem& p);
size_t split32_bytes(const Problem& p);
Split32 split32_layout(const Problem& p, void* base);
cudaError_t launch_tc_fwd32(const FwdArgs& a, const Split32& ws, cudaStream_t s);

// 3xTF32 tensor-core reverse pass for fp32 inputs (d = v = 64): a
// preparation kernel writes the tf32 hi / lo parts of Q, dY, K, V (and of Q,
// dY, K transposed) to the workspace, then a query-major dQ kernel and a
// key-major dK / dV kernel.  delta and L log2(e) must be in place (launch_delta).
struct Bwd32Split {
  float *qh, *ql, *yh, *yl;      // [BH][n][64]
  float *kh, *kl, *vh, *vl;      // [BH][nk][64]
  float *qth, *qtl, *yth, *ytl;  // [BH][64][ldq]
  float *kth, *ktl;              // [BH][64][ldk]
  int ldq, ldk;                  // n, nk rounded up to 32
  size_t bytes;
};
bool tc_bwd32_supported(const Problem& p);
size_t bwd32_bytes(const Problem& p);
Bwd32Split bwd32_layout(const Problem& p, void* base);
cudaError_t launch_tc_bwd32(const BwdArgs& a, const Bwd32Split& w, cudaStream_t s);

// Split-KV forward (nq queries aligned to the end of nk keys).
struct SplitArgs {
  const void* Q;
  const void* K;
  const void* V;
  int BH, nq, nk, d, v, mask_kind, window, words_per_row, splits, chunk;
  const uint32_t* bits;  // [nq][ceil(nk/32)]
  float sl2;             // scale * log2(e)
  float* pm;             // [BH][splits][nq] running max (exp2 domain)
  float* pl;             // [BH][splits][nq] running sum
  float* pz;             // [BH][splits][nq][v] unnormalised output
  unsigned* counters;    // [BH] chunks finished (zeroed before the launch)
  void* Y;               // outputs, for the kernels that merge in their last CTA
  float* L;
  unsigned* status;
};
size_t splitkv_smem_bytes(int nq, int d, int v, int elem_bytes);
int splitkv_max_queries();
int splitkv_reg_max_queries();  // nq up to this runs the register-resident chunk kernel
cudaError_t launch_splitkv(const SplitArgs& a, int dtype, void* Y, float* L, unsigned* status,
                           cudaStream_t s);
// The star merge of the chunk summaries alone (after launch_tc_fwd_chunks).
cudaError_t launch_splitkv_merge(const SplitArgs& a, int dtype, void* Y, float* L,
                                 unsigned* status, cudaStream_t s);

}  // namespace exattn
