// The C ABI of libexattn (include/exattn.h): argument checks, workspace layout
// and kernel dispatch.  No memory is allocated here.
#include <algorithm>
#include <math.h>
#include <stdint.h>
#include <stdio.h>

#include <atomic>

#include "../../include/exattn.h"
#include "internal.h"

namespace {

using namespace exattn;

std::atomic<int> g_path{EXATTN_PATH_AUTO};
std::atomic<unsigned long long> g_launches{0};
std::atomic<void*> g_hook_start[kKernRoles];
std::atomic<void*> g_hook_stop[kKernRoles];

constexpr int kMaxWidth = 256;
constexpr int kMaxN = 1 << 20;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Problem dimensions of either shape struct (nq == nk for exattn_shape).
struct Dims {
  int batch, heads, nq, nk, d, v, dtype;
};
Dims dims_of(const exattn_shape* s) { return {s->batch, s->heads, s->n, s->n, s->d, s->v, s->dtype}; }
Dims dims_of(const exattn_qk_shape* s) {
  return {s->batch, s->heads, s->nq, s->nk, s->d, s->v, s->dtype};
}

int check_dims(const Dims& s) {
  if (s.batch < 1 || s.heads < 1 || s.nq < 1 || s.nk < 1 || s.d < 1 || s.v < 1)
    return EXATTN_INVALID_ARG;
  if (s.dtype != EXATTN_F32 && s.dtype != EXATTN_BF16) return EXATTN_INVALID_ARG;
  if (s.d > kMaxWidth || s.v > kMaxWidth || s.nq > kMaxN || s.nk > kMaxN)
    return EXATTN_UNSUPPORTED;
  if ((long long)s.batch * s.heads > 65535) return EXATTN_UNSUPPORTED;
  if (s.dtype == EXATTN_BF16 && (s.d % 8 != 0 || s.v % 8 != 0)) return EXATTN_UNSUPPORTED;
  return EXATTN_OK;
}

int check_shape(const exattn_shape* s) { return s ? check_dims(dims_of(s)) : EXATTN_INVALID_ARG; }

int check_mask(int mask_kind, int window, const uint32_t* bitmask) {
  if (mask_kind < EXATTN_MASK_NONE || mask_kind > EXATTN_MASK_BITMASK) return EXATTN_INVALID_ARG;
  if (mask_kind == EXATTN_MASK_WINDOW && window < 1) return EXATTN_INVALID_ARG;
  if (mask_kind == EXATTN_MASK_BITMASK && bitmask == nullptr) return EXATTN_INVALID_ARG;
  if (mask_kind == EXATTN_MASK_BITMASK && (reinterpret_cast<uintptr_t>(bitmask) & 3u))
    return EXATTN_MISALIGNED;
  return EXATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

Problem make_problem(const Dims& s, float scale, int mask_kind, int window,
                     const uint32_t* bitmask) {
  Problem p;
  p.BH = s.batch * s.heads;
  p.n = s.nq;
  p.nk = s.nk;
  p.d = s.d;
  p.v = s.v;
  p.dtype = s.dtype;
  p.scale = scale;
  p.mask_kind = mask_kind;
  p.window = mask_kind == EXATTN_MASK_WINDOW ? window : 0;
  p.words_per_row = (s.nk + 31) / 32;
  p.bitmask = mask_kind == EXATTN_MASK_BITMASK ? bitmask : nullptr;
  p.drop_t = 0;
  p.drop_scale = 1.f;
  p.seed_lo = p.seed_hi = 0;
  return p;
}

// Dropout threshold of a drop probability q in [0, 1): t = min(65535,
// floor(q * 65536 + 1/2)); kept entries are scaled by 65536 / (65536 - t).
bool valid_dropout(float q) { return q >= 0.f && q < 1.f; }  // false for NaN

void set_dropout(Problem& p, float q, uint64_t seed) {
  const double t = floor(static_cast<double>(q) * 65536.0 + 0.5);
  p.drop_t = t > 65535.0 ? 65535u : static_cast<uint32_t>(t);
  p.drop_scale = static_cast<float>(65536.0 / (65536.0 - p.drop_t));
  p.seed_lo = static_cast<uint32_t>(seed & 0xFFFFFFFFu);
  p.seed_hi = static_cast<uint32_t>(seed >> 32);
}

// Reverse-pass workspace: status word | delta [BH][npad] | lse2 [BH][npad] |
// dQ accumulator [BH][nq][d] (fp32), each part 256-byte aligned (npad: nq
// rounded up to 128).
size_t npad_of(const Dims& s) { return ((size_t)s.nq + 127) / 128 * 128; }
size_t bwd_vec_bytes(const Dims& s) {
  return align_up(sizeof(float) * (size_t)s.batch * s.heads * npad_of(s), 256);
}
size_t bwd_delta_offset() { return kStatusBytes; }
size_t bwd_lse2_offset(const Dims& s) { return kStatusBytes + bwd_vec_bytes(s); }
size_t bwd_dqacc_offset(const Dims& s) { return kStatusBytes + 2 * bwd_vec_bytes(s); }
size_t bwd_bwd32_offset(const Dims& s) {
  return align_up(bwd_dqacc_offset(s) + sizeof(float) * (size_t)s.batch * s.heads * s.nq * s.d,
                  256);
}
// fp32 with d = v = 64 (the 3xTF32 reverse pass) also holds the tf32 parts of
// Q, dY, K, V after the accumulator.
bool bwd32_shape(const Dims& s) { return s.dtype == EXATTN_F32 && s.d == 64 && s.v == 64; }
size_t bwd_ws_bytes(const Dims& s) {
  if (!bwd32_shape(s))
    return bwd_dqacc_offset(s) + sizeof(float) * (size_t)s.batch * s.heads * s.nq * s.d;
  return bwd_bwd32_offset(s) +
         bwd32_bytes(make_problem(s, 1.f, EXATTN_MASK_NONE, 0, nullptr));
}

}  // namespace

namespace exattn {

thread_local char g_last_error[256] = "";

void record_error(const char* where, int code, const char* detail) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %d (%s)", where, code, detail ? detail : "");
}

void before_launch(int role, cudaStream_t s) {
  g_launches.fetch_add(1);
  void* ev = g_hook_start[role].exchange(nullptr);
  if (ev) cudaEventRecord(static_cast<cudaEvent_t>(ev), s);
}

void after_launch(int role, cudaStream_t s) {
  void* ev = g_hook_stop[role].exchange(nullptr);
  if (ev) cudaEventRecord(static_cast<cudaEvent_t>(ev), s);
}

}  // namespace exattn

extern "C" {

int exattn_record_kernel_events(int which, void* start, void* stop) {
  if (which < 0 || which >= kKernRoles) return -1;
  g_hook_start[which].store(start);
  g_hook_stop[which].store(stop);
  return 0;
}

unsigned long long exattn_launch_count(void) { return g_launches.load(); }

const char* exattn_last_error(void) { return g_last_error; }

namespace {
int cuda_status(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return EXATTN_OK;
  if (exattn::g_last_error[0] == 0 || e != cudaErrorInvalidValue)
    exattn::record_error(where, static_cast<int>(e), cudaGetErrorString(e));
  return EXATTN_CUDA_ERROR;
}
}  // namespace


int exattn_set_path(int path) {
  if (path != EXATTN_PATH_AUTO && path != EXATTN_PATH_SIMT && path != EXATTN_PATH_ATOMIC_DQ)
    return -1;
  return g_path.exchange(path);
}

// Forward workspace: the status word, plus for fp32 shapes that the 3xTF32
// tensor-core forward takes (d, v <= 128, multiples of 4) the split copies of K and V.
static size_t fwd_ws_bytes(const Dims& s) {
  if (s.dtype != EXATTN_F32 || !tc_fwd32_shape(s.d, s.v)) return kStatusBytes;
  Problem p = make_problem(s, 1.f, EXATTN_MASK_NONE, 0, nullptr);
  return kStatusBytes + split32_bytes(p);
}

size_t exattn_fwd_workspace_size(const exattn_shape* shape, int mask_kind) {
  if (check_shape(shape) != EXATTN_OK) return 0;
  (void)mask_kind;
  return fwd_ws_bytes(dims_of(shape));
}

size_t exattn_bwd_workspace_size(const exattn_shape* shape, int mask_kind) {
  if (check_shape(shape) != EXATTN_OK) return 0;
  (void)mask_kind;
  return bwd_ws_bytes(dims_of(shape));
}

size_t exattn_fwd_qk_workspace_size(const exattn_qk_shape* shape, int mask_kind) {
  if (!shape || check_dims(dims_of(shape)) != EXATTN_OK) return 0;
  (void)mask_kind;
  return fwd_ws_bytes(dims_of(shape));
}

size_t exattn_bwd_qk_workspace_size(const exattn_qk_shape* shape, int mask_kind) {
  if (!shape || check_dims(dims_of(shape)) != EXATTN_OK) return 0;
  (void)mask_kind;
  return bwd_ws_bytes(dims_of(shape));
}

namespace {

int fwd_impl(const Dims& dims, const void* Q, const void* K, const void* V, float scale,
             int mask_kind, int window, const uint32_t* bitmask, float dropout_p, uint64_t seed,
             void* Y, float* L, void* workspace, size_t workspace_bytes, void* cuda_stream) {
  int st = check_dims(dims);
  if (st != EXATTN_OK) return st;
  st = check_mask(mask_kind, window, bitmask);
  if (st != EXATTN_OK) return st;
  if (!valid_dropout(dropout_p)) return EXATTN_INVALID_ARG;
  if (!Q || !K || !V || !Y || !L || !workspace) return EXATTN_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(Y) || !aligned16(L))
    return EXATTN_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return EXATTN_MISALIGNED;
  if (workspace_bytes < fwd_ws_bytes(dims)) return EXATTN_WORKSPACE_TOO_SMALL;

  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  exattn::g_last_error[0] = 0;
  FwdArgs a;
  a.p = make_problem(dims, scale, mask_kind, window, bitmask);
  if (dropout_p > 0.f) set_dropout(a.p, dropout_p, seed);
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.Y = Y;
  a.L = L;
  a.status = static_cast<unsigned*>(workspace);
  cudaError_t e = cudaMemsetAsync(workspace, 0, kStatusBytes, s);
  if (e != cudaSuccess) return cuda_status(e, "attn_fwd: clearing the status word");
  if (g_path.load() != EXATTN_PATH_SIMT && tc_fwd_supported(a.p))
    return cuda_status(launch_tc_fwd(a, s), "attn_fwd: tensor-core forward launch");
  if (g_path.load() != EXATTN_PATH_SIMT && tc_fwd32_supported(a.p))
    return cuda_status(
        launch_tc_fwd32(a, split32_layout(a.p, static_cast<char*>(workspace) + kStatusBytes), s),
        "attn_fwd: 3xTF32 forward launch");
  return cuda_status(launch_simt_fwd(a, s), "attn_fwd: SIMT forward launch");
}

int bwd_impl(const Dims& dims, const void* Q, const void* K, const void* V, const void* Y,
             const void* dY, const float* L, float scale, int mask_kind, int window,
             const uint32_t* bitmask, float dropout_p, uint64_t seed, void* dQ, void* dK,
             void* dV, void* workspace, size_t workspace_bytes, void* cuda_stream) {
  int st = check_dims(dims);
  if (st != EXATTN_OK) return st;
  st = check_mask(mask_kind, window, bitmask);
  if (st != EXATTN_OK) return st;
  if (!valid_dropout(dropout_p)) return EXATTN_INVALID_ARG;
  if (!Q || !K || !V || !Y || !dY || !L || !dQ || !dK || !dV || !workspace)
    return EXATTN_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(Y) || !aligned16(dY) ||
      !aligned16(L) || !aligned16(dQ) || !aligned16(dK) || !aligned16(dV))
    return EXATTN_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return EXATTN_MISALIGNED;
  if (workspace_bytes < bwd_ws_bytes(dims)) return EXATTN_WORKSPACE_TOO_SMALL;

  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  exattn::g_last_error[0] = 0;
  char* ws = static_cast<char*>(workspace);
  BwdArgs a;
  a.p = make_problem(dims, scale, mask_kind, window, bitmask);
  if (dropout_p > 0.f) set_dropout(a.p, dropout_p, seed);
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.Y = Y;
  a.dY = dY;
  a.L = L;
  a.dQ = dQ;
  a.dK = dK;
  a.dV = dV;
  a.status = reinterpret_cast<unsigned*>(ws);
  a.npad = static_cast<int>(npad_of(dims));
  a.delta = reinterpret_cast<float*>(ws + bwd_delta_offset());
  a.lse2 = reinterpret_cast<float*>(ws + bwd_lse2_offset(dims));
  a.dQacc = reinterpret_cast<float*>(ws + bwd_dqacc_offset(dims));
  const size_t acc_bytes = sizeof(float) * (size_t)a.p.BH * a.p.n * a.p.d;
  cudaError_t e = cudaMemsetAsync(ws, 0, kStatusBytes, s);
  if (e != cudaSuccess) return cuda_status(e, "attn_bwd: clearing the status word");
  const int path = g_path.load();
  if (path == EXATTN_PATH_AUTO && bwd32_shape(dims) && tc_bwd32_supported(a.p)) {
    // 3xTF32: delta and L log2(e), then the split of the operands, the dQ and
    // the dK / dV kernels; dQ is written directly.
    e = launch_delta(a, s);
    if (e != cudaSuccess) return cuda_status(e, "attn_bwd: delta launch");
    return cuda_status(launch_tc_bwd32(a, bwd32_layout(a.p, ws + bwd_bwd32_offset(dims)), s),
                       "attn_bwd: 3xTF32 reverse launch");
  }
  if (path == EXATTN_PATH_AUTO && tc_bwd_split_supported(a.p)) {
    // Split form: dQ is written directly, no accumulator; the dQ kernel also
    // forms delta and L log2(e).
    return cuda_status(launch_tc_bwd_split(a, s), "attn_bwd: reverse kernel launch");
  }
  e = cudaMemsetAsync(a.dQacc, 0, acc_bytes, s);
  if (e != cudaSuccess) return cuda_status(e, "attn_bwd: clearing the dQ accumulator");
  e = launch_delta(a, s);
  if (e != cudaSuccess) return cuda_status(e, "attn_bwd: delta launch");
  if (path != EXATTN_PATH_SIMT && tc_bwd_supported(a.p))
    e = launch_tc_bwd(a, s);
  else
    e = launch_simt_bwd(a, s);
  if (e != cudaSuccess) return cuda_status(e, "attn_bwd: reverse kernel launch");
  return cuda_status(launch_dq_convert(a, s), "attn_bwd: dQ conversion launch");
}

}  // namespace

int attn_fwd(const exattn_shape* shape, const void* Q, const void* K, const void* V,
             float scale, int mask_kind, int window, const uint32_t* bitmask, void* Y, float* L,
             void* workspace, size_t workspace_bytes, void* cuda_stream) {
  if (!shape) return EXATTN_INVALID_ARG;
  return fwd_impl(dims_of(shape), Q, K, V, scale, mask_kind, window, bitmask, 0.f, 0, Y, L,
                  workspace, workspace_bytes, cuda_stream);
}

int attn_fwd_dropout(const exattn_shape* shape, const void* Q, const void* K, const void* V,
                     float scale, int mask_kind, int window, const uint32_t* bitmask,
                     float dropout_p, uint64_t seed, void* Y, float* L, void* workspace,
                     size_t workspace_bytes, void* cuda_stream) {
  if (!shape) return EXATTN_INVALID_ARG;
  return fwd_impl(dims_of(shape), Q, K, V, scale, mask_kind, window, bitmask, dropout_p, seed, Y,
                  L, workspace, workspace_bytes, cuda_stream);
}

int attn_fwd_qk(const exattn_qk_shape* shape, const void* Q, const void* K, const void* V,
                float scale, int mask_kind, int window, const uint32_t* bitmask, float dropout_p,
                uint64_t seed, void* Y, float* L, void* workspace, size_t workspace_bytes,
                void* cuda_stream) {
  if (!shape) return EXATTN_INVALID_ARG;
  return fwd_impl(dims_of(shape), Q, K, V, scale, mask_kind, window, bitmask, dropout_p, seed, Y,
                  L, workspace, workspace_bytes, cuda_stream);
}

int attn_bwd(const exattn_shape* shape, const void* Q, const void* K, const void* V,
             const void* Y, const void* dY, const float* L, float scale, int mask_kind,
             int window, const uint32_t* bitmask, void* dQ, void* dK, void* dV, void* workspace,
             size_t workspace_bytes, void* cuda_stream) {
  if (!shape) return EXATTN_INVALID_ARG;
  return bwd_impl(dims_of(shape), Q, K, V, Y, dY, L, scale, mask_kind, window, bitmask, 0.f, 0,
                  dQ, dK, dV, workspace, workspace_bytes, cuda_stream);
}

int attn_bwd_dropout(const exattn_shape* shape, const void* Q, const void* K, const void* V,
                     const void* Y, const void* dY, const float* L, float scale, int mask_kind,
                     int window, const uint32_t* bitmask, float dropout_p, uint64_t seed,
                     void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                     void* cuda_stream) {
  if (!shape) return EXATTN_INVALID_ARG;
  return bwd_impl(dims_of(shape), Q, K, V, Y, dY, L, scale, mask_kind, window, bitmask,
                  dropout_p, seed, dQ, dK, dV, workspace, workspace_bytes, cuda_stream);
}

int attn_bwd_qk(const exattn_qk_shape* shape, const void* Q, const void* K, const void* V,
                const void* Y, const void* dY, const float* L, float scale, int mask_kind,
                int window, const uint32_t* bitmask, float dropout_p, uint64_t seed, void* dQ,
                void* dK, void* dV, void* workspace, size_t workspace_bytes, void* cuda_stream) {
  if (!shape) return EXATTN_INVALID_ARG;
  return bwd_impl(dims_of(shape), Q, K, V, Y, dY, L, scale, mask_kind, window, bitmask,
                  dropout_p, seed, dQ, dK, dV, workspace, workspace_bytes, cuda_stream);
}

namespace {

int check_qk_shape(const exattn_qk_shape* s) {
  if (!s) return EXATTN_INVALID_ARG;
  if (s->batch < 1 || s->heads < 1 || s->nq < 1 || s->nk < 1 || s->d < 1 || s->v < 1)
    return EXATTN_INVALID_ARG;
  if (s->dtype != EXATTN_F32 && s->dtype != EXATTN_BF16) return EXATTN_INVALID_ARG;
  if (s->nq > splitkv_max_queries() || s->d > kMaxWidth || s->v > kMaxWidth || s->nk > kMaxN)
    return EXATTN_UNSUPPORTED;
  if ((long long)s->batch * s->heads > 65535) return EXATTN_UNSUPPORTED;
  // K and V rows are staged in 16-byte pieces.
  const int per16 = s->dtype == EXATTN_BF16 ? 8 : 4;
  if (s->d % per16 != 0 || s->v % per16 != 0) return EXATTN_UNSUPPORTED;
  if (splitkv_smem_bytes(s->nq, s->d, s->v, s->dtype == EXATTN_BF16 ? 2 : 4) > 200 * 1024)
    return EXATTN_UNSUPPORTED;
  return EXATTN_OK;
}

// Shapes whose chunks can run on the tensor-core forward in summary mode
// (bf16, d = v in {64, 128}, two or more queries).  A single query stays on the
// register kernel, which streams K and V near the copy bandwidth; from two
// queries on, the register kernel's per-lane state leaves it too few loads in
// flight, while the tensor-core chunks stream K and V through TMA whatever nq.
// The plan depends on the shape alone, so the workspace query and the call
// agree whatever the kernel path setting.
bool splitkv_tc_shape(const exattn_qk_shape* s) {
  return s->dtype == EXATTN_BF16 && s->d == s->v && (s->d == 64 || s->d == 128) && s->nq > 1;
}

// num_splits == 0: enough chunks for about 8 waves of resident CTAs over all
// batch*head slices (the register kernel keeps 4 CTAs per SM of the 152-SM
// part, the tensor-core kernel 1), with at least 256 keys per chunk.
constexpr int kAutoMinChunk = 256;

int resolve_splits(const exattn_qk_shape* s, int num_splits) {
  if (num_splits != 0) return num_splits;
  const int target = (splitkv_tc_shape(s) ? 8 : 32) * 152;
  const int bh = s->batch * s->heads;
  const int want = (target + bh - 1) / bh;
  const int most = (s->nk + kAutoMinChunk - 1) / kAutoMinChunk;
  return want < 1 ? 1 : (want > most ? most : want);
}

// Keys per chunk (a multiple of 32, of 128 for tensor-core shapes) and the
// number of chunks actually used.
void split_plan(const exattn_qk_shape* s, int num_splits, int* chunk, int* splits) {
  const int gran = splitkv_tc_shape(s) ? 128 : 32;
  int c = (s->nk + num_splits - 1) / num_splits;
  c = (c + gran - 1) / gran * gran;
  *chunk = c;
  *splits = (s->nk + c - 1) / c;
}

}  // namespace

size_t exattn_splitkv_workspace_size(const exattn_qk_shape* shape, int num_splits) {
  if (check_qk_shape(shape) != EXATTN_OK || num_splits < 0 || num_splits > 4096) return 0;
  num_splits = resolve_splits(shape, num_splits);
  int chunk, splits;
  split_plan(shape, num_splits, &chunk, &splits);
  const size_t bh = (size_t)shape->batch * shape->heads;
  const size_t rows = bh * splits * shape->nq;
  return kStatusBytes + align_up(sizeof(unsigned) * bh, 256) +
         2 * align_up(sizeof(float) * rows, 256) + sizeof(float) * rows * shape->v;
}

int attn_fwd_splitkv(const exattn_qk_shape* shape, const void* Q, const void* K, const void* V,
                     float scale, int mask_kind, int window, const uint32_t* bitmask,
                     int num_splits, void* Y, float* L, void* workspace, size_t workspace_bytes,
                     void* cuda_stream) {
  int st = check_qk_shape(shape);
  if (st != EXATTN_OK) return st;
  st = check_mask(mask_kind, window, bitmask);
  if (st != EXATTN_OK) return st;
  if (num_splits < 0 || num_splits > 4096) return EXATTN_INVALID_ARG;
  if (!Q || !K || !V || !Y || !L || !workspace) return EXATTN_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(Y) || !aligned16(L))
    return EXATTN_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return EXATTN_MISALIGNED;
  if (workspace_bytes < exattn_splitkv_workspace_size(shape, num_splits))
    return EXATTN_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  exattn::g_last_error[0] = 0;
  SplitArgs a;
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.BH = shape->batch * shape->heads;
  a.nq = shape->nq;
  a.nk = shape->nk;
  a.d = shape->d;
  a.v = shape->v;
  a.mask_kind = mask_kind;
  a.window = mask_kind == EXATTN_MASK_WINDOW ? window : 0;
  a.words_per_row = (shape->nk + 31) / 32;
  a.bits = mask_kind == EXATTN_MASK_BITMASK ? bitmask : nullptr;
  a.sl2 = scale * 1.4426950408889634f;
  split_plan(shape, resolve_splits(shape, num_splits), &a.chunk, &a.splits);
  // Workspace: status word | chunk counters [BH] | m | l | z (each 256-byte aligned).
  const size_t rows = (size_t)a.BH * a.splits * a.nq;
  const size_t cnt_bytes = align_up(sizeof(unsigned) * a.BH, 256);
  char* ws = static_cast<char*>(workspace) + kStatusBytes;
  a.counters = reinterpret_cast<unsigned*>(ws);
  ws += cnt_bytes;
  a.pm = reinterpret_cast<float*>(ws);
  a.pl = reinterpret_cast<float*>(ws + align_up(sizeof(float) * rows, 256));
  a.pz = reinterpret_cast<float*>(ws + 2 * align_up(sizeof(float) * rows, 256));
  a.Y = Y;
  a.L = L;
  a.status = static_cast<unsigned*>(workspace);
  cudaError_t e = cudaMemsetAsync(workspace, 0, kStatusBytes + cnt_bytes, s);
  if (e != cudaSuccess) return cuda_status(e, "attn_fwd_splitkv: clearing the status word");
  if (g_path.load() != EXATTN_PATH_SIMT && splitkv_tc_shape(shape)) {
    // Chunks on the tensor-core forward in summary mode, then the merge.
    FwdArgs f;
    f.p = make_problem(dims_of(shape), scale, mask_kind, window, bitmask);
    if (tc_fwd_supported(f.p)) {
      f.Q = Q;
      f.K = K;
      f.V = V;
      f.Y = Y;
      f.L = L;
      f.status = a.status;
      e = launch_tc_fwd_chunks(f, a.chunk, a.splits, a.pm, a.pl, a.pz, s);
      if (e != cudaSuccess) return cuda_status(e, "attn_fwd_splitkv: tensor-core chunks");
      return cuda_status(launch_splitkv_merge(a, shape->dtype, Y, L, a.status, s),
                         "attn_fwd_splitkv: merge launch");
    }
  }
  return cuda_status(launch_splitkv(a, shape->dtype, Y, L, static_cast<unsigned*>(workspace), s),
                     "attn_fwd_splitkv: launch");
}

// ------------------------------------------------------------ host step
// attn_step_host: forward and reverse pass on tensors in host memory.  The
// slices are cut into chunks; chunk k's inputs are copied in on one stream,
// its forward and reverse pass run on a second, and its outputs are copied out
// on a third, so the copies of neighbouring chunks overlap the kernels.  Each
// slice is computed exactly as attn_fwd / attn_bwd compute it.
}  // extern "C"

namespace {

__global__ void status_or_kernel(unsigned* dst, const unsigned* src) { *dst |= *src; }

constexpr int kHostMaxChunks = 16;

struct HostStepLayout {
  int chunks;
  int start[kHostMaxChunks + 1];  // chunk c holds slices [start[c], start[c + 1])
  size_t q, k, v, dy, y, l, dq, dk, dv, bits, ws, ws_bytes, total;
};

HostStepLayout host_layout(const Dims& d, int mask_kind) {
  HostStepLayout L{};
  const int BH = d.batch * d.heads;
  const size_t e = d.dtype == EXATTN_F32 ? 4 : 2;
  const size_t row_q = (size_t)d.d * e, row_v = (size_t)d.v * e;
  // Chunk boundaries must keep every slice pointer 16-byte aligned.
  const bool split_ok = ((size_t)d.nq * row_q) % 16 == 0 && ((size_t)d.nq * row_v) % 16 == 0 &&
                        ((size_t)d.nq * 4) % 16 == 0;
  // Nothing computes until the first chunk is in and the last chunk's outputs
  // leave after everything else, so those two are small (1/32 of the slices
  // each) and the middle is cut evenly.
  L.chunks = 1;
  L.start[0] = 0;
  L.start[1] = BH;
  if (split_ok && BH >= 8) {
    const int edge = BH >= 64 ? BH / 32 : 0;
    const int middle = BH >= 64 ? 6 : 4;
    int c = 0;
    if (edge > 0) L.start[++c] = edge;
    const int m0 = L.start[c], m1 = BH - edge;
    for (int k = 1; k <= middle; ++k) L.start[++c] = m0 + (int)((long long)(m1 - m0) * k / middle);
    if (edge > 0) L.start[++c] = BH;
    L.chunks = c;
  }
  int per = 0;
  for (int c = 0; c < L.chunks; ++c) per = std::max(per, L.start[c + 1] - L.start[c]);
  size_t o = kStatusBytes;  // the step's status word (OR of the chunks') and padding
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  const size_t slice_q = (size_t)d.nq * row_q, slice_v = (size_t)d.nq * row_v;
  L.q = take(BH * slice_q);
  L.k = take(BH * slice_q);
  L.v = take(BH * slice_v);
  L.dy = take(BH * slice_v);
  L.y = take(BH * slice_v);
  L.l = take((size_t)BH * d.nq * 4);
  L.dq = take(BH * slice_q);
  L.dk = take(BH * slice_q);
  L.dv = take(BH * slice_v);
  L.bits = take(mask_kind == kMaskBitmask ? (size_t)d.nq * ((d.nk + 31) / 32) * 4 : 0);
  const Dims c{1, per, d.nq, d.nk, d.d, d.v, d.dtype};
  L.ws_bytes = std::max(fwd_ws_bytes(c), bwd_ws_bytes(c));
  L.ws = take(L.ws_bytes);
  L.total = o;
  return L;
}

// Streams and events of the host step, made once per host thread and device
// and released when the thread exits (or right away if making one of them
// fails).  Destroying a stream or event whose work is still queued is allowed:
// CUDA releases it once that work completes.  At process exit the runtime may
// already be unloading; the calls then fail harmlessly.
constexpr int kHostMaxDevices = 64;
struct HostStepStreams {
  int device = -1;
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, loaded[kHostMaxChunks] = {}, done[kHostMaxChunks] = {},
              end_in = nullptr, end_comp = nullptr, end_out = nullptr;

  HostStepStreams() = default;
  HostStepStreams(const HostStepStreams&) = delete;
  HostStepStreams& operator=(const HostStepStreams&) = delete;
  ~HostStepStreams() { release(); }

  // Destroys whatever was made, on the device it was made on.
  void release() {
    if (device < 0) return;
    int cur = -1;
    const bool switched = cudaGetDevice(&cur) == cudaSuccess && cur != device &&
                          cudaSetDevice(device) == cudaSuccess;
    for (cudaStream_t* st : {&in, &comp, &out})
      if (*st) {
        cudaStreamDestroy(*st);
        *st = nullptr;
      }
    for (cudaEvent_t* ev : {&start, &end_in, &end_comp, &end_out})
      if (*ev) {
        cudaEventDestroy(*ev);
        *ev = nullptr;
      }
    for (int c = 0; c < kHostMaxChunks; ++c)
      for (cudaEvent_t* ev : {&loaded[c], &done[c]})
        if (*ev) {
          cudaEventDestroy(*ev);
          *ev = nullptr;
        }
    if (switched) cudaSetDevice(cur);
    device = -1;
  }

  // Makes every stream and event on the current device `dev`; on failure
  // releases those already made and returns the error.
  cudaError_t create(int dev) {
    device = dev;
    const unsigned f = cudaEventDisableTiming;
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&comp, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&start, f)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&end_in, f)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&end_comp, f)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&end_out, f)) != cudaSuccess) {
      release();
      return e;
    }
    for (int c = 0; c < kHostMaxChunks; ++c)
      if ((e = cudaEventCreateWithFlags(&loaded[c], f)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&done[c], f)) != cudaSuccess) {
        release();
        return e;
      }
    return cudaSuccess;
  }
};

cudaError_t host_streams(HostStepStreams*& hs) {
  thread_local HostStepStreams caches[kHostMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kHostMaxDevices) return cudaErrorInvalidDevice;
  HostStepStreams& cache = caches[dev];
  if (cache.device != dev && (e = cache.create(dev)) != cudaSuccess) return e;
  hs = &cache;
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t exattn_host_step_workspace_size(const exattn_shape* shape, int mask_kind) {
  if (check_shape(shape) != EXATTN_OK) return 0;
  return host_layout(dims_of(shape), mask_kind).total;
}

int attn_step_host(const exattn_shape* shape, const void* Q, const void* K, const void* V,
                   const void* dY, float scale, int mask_kind, int window, const uint32_t* bitmask,
                   void* Y, float* L, void* dQ, void* dK, void* dV, void* workspace,
                   size_t workspace_bytes, void* cuda_stream) {
  int st = check_shape(shape);
  if (st != EXATTN_OK) return st;
  st = check_mask(mask_kind, window, bitmask);
  if (st != EXATTN_OK) return st;
  if (!Q || !K || !V || !dY || !Y || !L || !dQ || !dK || !dV || !workspace)
    return EXATTN_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return EXATTN_MISALIGNED;
  const Dims d = dims_of(shape);
  const HostStepLayout lay = host_layout(d, mask_kind);
  if (workspace_bytes < lay.total) return EXATTN_WORKSPACE_TOO_SMALL;
  exattn::g_last_error[0] = 0;
  HostStepStreams* hs = nullptr;
  cudaError_t e = host_streams(hs);
  if (e != cudaSuccess) return cuda_status(e, "attn_step_host: streams");
  cudaStream_t user = static_cast<cudaStream_t>(cuda_stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t es = d.dtype == EXATTN_F32 ? 4 : 2;
  const size_t sq = (size_t)d.nq * d.d * es, sv = (size_t)d.nq * d.v * es, sl = (size_t)d.nq * 4;
  // Everything after the work already queued on the caller's stream.
  if ((e = cudaMemsetAsync(ws, 0, kStatusBytes, user)) != cudaSuccess ||
      (e = cudaEventRecord(hs->start, user)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hs->in, hs->start, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hs->comp, hs->start, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hs->out, hs->start, 0)) != cudaSuccess)
    return cuda_status(e, "attn_step_host: ordering");
  // The copies and kernels of every chunk.  Whatever it returns, the caller's
  // stream then waits for all three internal streams, so no queued copy can
  // outlive the buffers the caller frees after a failure.
  auto queue = [&]() -> int {
    const uint32_t* bits_dev = nullptr;
    if (mask_kind == kMaskBitmask) {
      const size_t bytes = (size_t)d.nq * ((d.nk + 31) / 32) * 4;
      if ((e = cudaMemcpyAsync(ws + lay.bits, bitmask, bytes, cudaMemcpyHostToDevice, hs->in)) !=
          cudaSuccess)
        return cuda_status(e, "attn_step_host: bitmask copy");
      bits_dev = reinterpret_cast<const uint32_t*>(ws + lay.bits);
    }
    auto h2d = [&](size_t dev_off, const void* host, size_t off, size_t bytes) {
      return cudaMemcpyAsync(ws + dev_off + off, static_cast<const uint8_t*>(host) + off, bytes,
                             cudaMemcpyHostToDevice, hs->in);
    };
    auto d2h = [&](void* host, size_t dev_off, size_t off, size_t bytes) {
      return cudaMemcpyAsync(static_cast<uint8_t*>(host) + off, ws + dev_off + off, bytes,
                             cudaMemcpyDeviceToHost, hs->out);
    };
    for (int c = 0; c < lay.chunks; ++c) {
      const int s0 = lay.start[c], cnt = lay.start[c + 1] - s0;
      const size_t oq = s0 * sq, ov = s0 * sv, ol = s0 * sl;
      if ((e = h2d(lay.q, Q, oq, cnt * sq)) != cudaSuccess ||
          (e = h2d(lay.k, K, oq, cnt * sq)) != cudaSuccess ||
          (e = h2d(lay.v, V, ov, cnt * sv)) != cudaSuccess ||
          (e = h2d(lay.dy, dY, ov, cnt * sv)) != cudaSuccess ||
          (e = cudaEventRecord(hs->loaded[c % kHostMaxChunks], hs->in)) != cudaSuccess ||
          (e = cudaStreamWaitEvent(hs->comp, hs->loaded[c % kHostMaxChunks], 0)) != cudaSuccess)
        return cuda_status(e, "attn_step_host: input copies");
      const Dims cd{1, cnt, d.nq, d.nk, d.d, d.v, d.dtype};
      uint8_t* cws = ws + lay.ws;
      st = fwd_impl(cd, ws + lay.q + oq, ws + lay.k + oq, ws + lay.v + ov, scale, mask_kind, window,
                    bits_dev, 0.f, 0, ws + lay.y + ov, reinterpret_cast<float*>(ws + lay.l + ol),
                    cws, lay.ws_bytes, hs->comp);
      if (st != EXATTN_OK) return st;
      g_launches.fetch_add(1);
      status_or_kernel<<<1, 1, 0, hs->comp>>>(reinterpret_cast<unsigned*>(ws),
                                              reinterpret_cast<const unsigned*>(cws));
      st = bwd_impl(cd, ws + lay.q + oq, ws + lay.k + oq, ws + lay.v + ov, ws + lay.y + ov,
                    ws + lay.dy + ov, reinterpret_cast<const float*>(ws + lay.l + ol), scale,
                    mask_kind, window, bits_dev, 0.f, 0, ws + lay.dq + oq, ws + lay.dk + oq,
                    ws + lay.dv + ov, cws, lay.ws_bytes, hs->comp);
      if (st != EXATTN_OK) return st;
      g_launches.fetch_add(1);
      status_or_kernel<<<1, 1, 0, hs->comp>>>(reinterpret_cast<unsigned*>(ws),
                                              reinterpret_cast<const unsigned*>(cws));
      if ((e = cudaEventRecord(hs->done[c % kHostMaxChunks], hs->comp)) != cudaSuccess ||
          (e = cudaStreamWaitEvent(hs->out, hs->done[c % kHostMaxChunks], 0)) != cudaSuccess ||
          (e = d2h(Y, lay.y, ov, cnt * sv)) != cudaSuccess ||
          (e = d2h(L, lay.l, ol, cnt * sl)) != cudaSuccess ||
          (e = d2h(dQ, lay.dq, oq, cnt * sq)) != cudaSuccess ||
          (e = d2h(dK, lay.dk, oq, cnt * sq)) != cudaSuccess ||
          (e = d2h(dV, lay.dv, ov, cnt * sv)) != cudaSuccess)
        return cuda_status(e, "attn_step_host: output copies");
    }
    return EXATTN_OK;
  };
  const int queued = queue();
  // The caller's stream continues after the last copy out and the last kernel.
  if ((e = cudaEventRecord(hs->end_out, hs->out)) != cudaSuccess ||
      (e = cudaEventRecord(hs->end_comp, hs->comp)) != cudaSuccess ||
      (e = cudaEventRecord(hs->end_in, hs->in)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(user, hs->end_out, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(user, hs->end_comp, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(user, hs->end_in, 0)) != cudaSuccess)
    return queued != EXATTN_OK ? queued : cuda_status(e, "attn_step_host: ordering");
  return queued;
}

int exattn_device_status(const void* workspace, void* cuda_stream) {
  if (!workspace) return EXATTN_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return EXATTN_CUDA_ERROR;
  unsigned word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return EXATTN_CUDA_ERROR;
  if (word & 2u) return EXATTN_TIMEOUT;
  if (word & 1u) return EXATTN_EMPTY_ROW;
  return EXATTN_OK;
}

const char* exattn_status_string(int status) {
  switch (status) {
    case EXATTN_OK: return "ok";
    case EXATTN_INVALID_ARG: return "invalid argument";
    case EXATTN_UNSUPPORTED: return "unsupported shape";
    case EXATTN_MISALIGNED: return "misaligned pointer";
    case EXATTN_WORKSPACE_TOO_SMALL: return "workspace too small";
    case EXATTN_EMPTY_ROW: return "an allowed-key set was empty";
    case EXATTN_CUDA_ERROR: return "CUDA error";
    case EXATTN_TIMEOUT: return "a bounded device wait timed out";
    default: return "unknown status";
  }
}

}  // extern "C"
