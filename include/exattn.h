/*
 * exattn.h -- C ABI of libexattn.so: exact masked scaled-dot-product attention,
 * computed tile by tile on one GB300 GPU (sm_103a).
 *
 * The operation is the one stated in "Exact tiled softmax attention with
 * block-recomputed vector-Jacobian products" (alphabetamath), Inputs: matrices
 * Q, K in R^{n x d}, V in R^{n x v}, a real scale c, and nonempty allowed-key
 * sets A_1..A_n read on demand from caller-owned storage.  Per (batch, head):
 *
 *   s_ij = c <Q_i, K_j> (j in A_i),  p_ij = exp(s_ij - m_i) / l_i,
 *   Y_i  = sum_j p_ij V_j,           L_i = m_i + ln l_i  (natural log).
 *
 * attn_fwd runs the Forward procedure of that page (an online-softmax
 * recurrence over key blocks, whole blocks with I = J_t n A_i empty skipped)
 * and retains L_i, the statistic of "python-flash-attention-online-softmax-
 * block-recompute", The fix, item 1.  attn_bwd runs the Reverse procedure:
 * delta_i = G_i . Y_i (HarshvardhanJ/FlashAttention, backward section), then
 * per key block it recomputes p_ij from Q, K and the frozen L_i and adds
 *   dQ_i += c gamma_ij K_j,  dK_j += c gamma_ij Q_i,  dV_j += p_ij G_i,
 *   gamma_ij = p_ij (G_i . V_j - delta_i).
 * No n x n score or probability matrix is ever stored.
 *
 * Layout.  Every matrix is dense, contiguous, row-major, batched as
 * [batch][heads][n][width]: Q, K, dQ, dK are [B][H][n][d]; V, Y, dY, dV are
 * [B][H][n][v]; L is float32 [B][H][n].  Q, K, V, Y, dY, dQ, dK, dV have the
 * element type `dtype`; L is always float32.  Device pointers only (memory
 * the GPU can address), 16-byte aligned.
 *
 * Masks (0-indexed, one mask shared by every batch and head):
 *   EXATTN_MASK_NONE     A_i = {0 .. n-1}
 *   EXATTN_MASK_CAUSAL   A_i = {0 .. i}
 *   EXATTN_MASK_WINDOW   A_i = {max(0, i-window+1) .. i}, window >= 1
 *   EXATTN_MASK_BITMASK  j in A_i iff bit (j % 32) of bitmask[i*ceil(n/32) + j/32]
 *                        is set; `bitmask` is a device array of n*ceil(n/32)
 *                        uint32 words owned by the caller.
 *
 * Ownership and streams.  The caller owns every buffer, the workspace
 * included.  The library allocates no memory and keeps no pointer after a
 * call returns.  Work is queued on `cuda_stream` (a cudaStream_t; NULL is the
 * legacy default stream) and runs asynchronously; the return code covers
 * argument checks and kernel launches only.
 *
 * Aliasing.  Q, K and V may alias one another (self-attention, Q = K = V = X;
 * the caller then forms dX = dQ + dK + dV).  Outputs must not alias inputs or
 * each other.  Two calls that share a workspace must not overlap in time.
 *
 * Empty allowed sets.  A nonempty A_i is a precondition.  A row that breaks
 * it gets Y_i = 0 and L_i = -inf, contributes nothing to the gradients, and
 * the device status word of the workspace records EXATTN_EMPTY_ROW (read it
 * with exattn_device_status).  No NaN is produced.
 */
#ifndef EXATTN_H
#define EXATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types of Q, K, V, Y, dY, dQ, dK, dV. Accumulation is always fp32. */
enum exattn_dtype { EXATTN_F32 = 0, EXATTN_BF16 = 1 };

enum exattn_mask_kind {
  EXATTN_MASK_NONE = 0,
  EXATTN_MASK_CAUSAL = 1,
  EXATTN_MASK_WINDOW = 2,
  EXATTN_MASK_BITMASK = 3
};

/* Return codes.  Host-side checks return 1-4 and 6 before queuing any work;
 * 5 and 7 are device-side conditions reported through the status word. */
enum exattn_status {
  EXATTN_OK = 0,
  EXATTN_INVALID_ARG = 1,        /* null pointer, non-positive size, bad mask kind/window */
  EXATTN_UNSUPPORTED = 2,        /* d or v > 256, or bf16 with d or v not a multiple of 8 */
  EXATTN_MISALIGNED = 3,         /* a pointer is not 16-byte aligned */
  EXATTN_WORKSPACE_TOO_SMALL = 4,
  EXATTN_EMPTY_ROW = 5,          /* some A_i was empty (status word) */
  EXATTN_CUDA_ERROR = 6,         /* a CUDA call or launch failed */
  EXATTN_TIMEOUT = 7             /* a bounded wait inside a kernel gave up (status word) */
};

/* Problem shape.  batch, heads, n, d, v >= 1; dtype is an exattn_dtype. */
typedef struct exattn_shape {
  int batch;
  int heads;
  int n;
  int d;
  int v;
  int dtype;
} exattn_shape;

/* Kernel path selection, process-wide (default EXATTN_PATH_AUTO).
 * AUTO uses the tcgen05/TMA/TMEM kernels where the shape allows (bf16 with
 * d, v <= 128 and multiples of 8: widths other than 64 and 128 run on the
 * width-64 or width-128 kernels, whose TMA loads fill the missing columns with
 * zeros and whose stores leave them out; for fp32 with d, v <= 128 and multiples
 * of 4, a positive scale and no dropout the forward runs 3xTF32 on the tensor
 * cores, zero-padded the same way: each operand split into two tf32 parts,
 * three products per product, partial sums promoted to fp32 every key block;
 * the fp32 reverse pass runs 3xTF32 for d = v = 64 without dropout) and the
 * SIMT fp32 kernels otherwise (register-tiled for d, v <= 128 and multiples of
 * 4); the bf16 reverse pass is a key-major dK/dV kernel plus a query-major dQ
 * kernel.  SIMT forces the SIMT
 * kernels for every shape.  ATOMIC_DQ is AUTO with the other reverse form on
 * the tensor cores: one key-major kernel that adds dQ into an fp32 accumulator
 * with vector reductions (kept for measurement; bf16 d = v in {64, 128} only,
 * SIMT kernels otherwise).  Returns the previous
 * setting, or -1 for an unknown value (setting unchanged). */
enum exattn_path { EXATTN_PATH_AUTO = 0, EXATTN_PATH_SIMT = 1, EXATTN_PATH_ATOMIC_DQ = 2 };
int exattn_set_path(int path);

/* Workspace bytes that attn_fwd / attn_bwd need for this shape and mask kind.
 * The workspace holds the device status word (first 256 bytes); for an fp32
 * forward with d, v <= 128, multiples of 4 (the 3xTF32 tensor-core forward) also the
 * tf32 hi / lo split of K and V (4 copies of K's and V's size, V transposed
 * with rows padded to 32 keys); for the reverse pass delta [B][H][n], L log2(e)
 * [B][H][n] and the fp32 dQ accumulator [B][H][n][d].  Every size is linear in
 * n.  Returns 0 when the shape is invalid. */
size_t exattn_fwd_workspace_size(const exattn_shape* shape, int mask_kind);
size_t exattn_bwd_workspace_size(const exattn_shape* shape, int mask_kind);

/* Forward: Y [B][H][n][v] (dtype) and L [B][H][n] (float32, natural log) from
 * Q, K, V.  `window` is read for EXATTN_MASK_WINDOW only, `bitmask` for
 * EXATTN_MASK_BITMASK only (may be NULL otherwise).  `workspace` is a device
 * buffer of at least exattn_fwd_workspace_size bytes, 256-byte aligned; its
 * status word is cleared by the call.  Returns an exattn_status. */
int attn_fwd(const exattn_shape* shape, const void* Q, const void* K, const void* V,
             float scale, int mask_kind, int window, const uint32_t* bitmask,
             void* Y, float* L, void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Reverse pass for the upstream gradient dY (= G): writes dQ, dK (dtype,
 * [B][H][n][d]) and dV (dtype, [B][H][n][v]).  Y and L must come from attn_fwd
 * with the same Q, K, V, scale and mask.  A row whose L_i is -inf (its allowed
 * set was empty) contributes nothing, gets dQ_i = 0, and the status word of the
 * workspace records EXATTN_EMPTY_ROW.  `workspace` is a device buffer of at
 * least exattn_bwd_workspace_size bytes, 256-byte aligned.  Returns an
 * exattn_status. */
int attn_bwd(const exattn_shape* shape, const void* Q, const void* K, const void* V,
             const void* Y, const void* dY, const float* L, float scale, int mask_kind,
             int window, const uint32_t* bitmask, void* dQ, void* dK, void* dV,
             void* workspace, size_t workspace_bytes, void* cuda_stream);

/* ---------------------------------------------------------------------------
 * Dropout with a replayed mask.
 *
 * "Exact tiled softmax attention with block-recomputed vector-Jacobian
 * products", Reverse procedure: the base method has no dropout, and a dropout
 * extension must replay the forward pass's realised mask in its reverse pass.
 * Here the mask acts on the normalised probabilities:
 *   Y_i = sum_j p_ij xi_ij s V_j,   s = 65536 / (65536 - t),
 * with L_i the statistic of the undropped p (as in attn_fwd), and the reverse
 * pass uses the same xi:  dV_j += p_ij xi_ij s G_i,  dP_ij = xi_ij s G_i.V_j,
 * gamma_ij = p_ij (dP_ij - delta_i) with delta_i = G_i.Y_i.
 *
 * xi_ij is recomputed, never stored: key j of row i in slice bh = b*H + h is
 * kept when u_ij >= t, where t = min(65535, floor(dropout_p * 65536 + 1/2))
 * and u_ij is half (j % 2) (low half first) of word (j % 8) / 2 of the
 * Philox-4x32-10 output (Salmon et al., "Parallel random numbers: as easy as
 * 1, 2, 3", SC 2011) for counter (j / 8, i, bh, 0) and key (seed mod 2^32,
 * seed / 2^32).  The realised drop rate is t / 65536.
 *
 * Arguments as attn_fwd / attn_bwd plus dropout_p in [0, 1) (otherwise
 * EXATTN_INVALID_ARG) and the 64-bit seed; dropout_p = 0 is attn_fwd /
 * attn_bwd exactly.  attn_bwd_dropout must get the dropout_p and seed of the
 * attn_fwd_dropout call that produced Y and L.  Dropout runs on the tensor-core
 * kernels where attn_fwd / attn_bwd would (the atomic dQ form excepted: with
 * EXATTN_PATH_ATOMIC_DQ the reverse pass runs on the SIMT kernels).
 * ------------------------------------------------------------------------- */
int attn_fwd_dropout(const exattn_shape* shape, const void* Q, const void* K, const void* V,
                     float scale, int mask_kind, int window, const uint32_t* bitmask,
                     float dropout_p, uint64_t seed, void* Y, float* L, void* workspace,
                     size_t workspace_bytes, void* cuda_stream);
int attn_bwd_dropout(const exattn_shape* shape, const void* Q, const void* K, const void* V,
                     const void* Y, const void* dY, const float* L, float scale, int mask_kind,
                     int window, const uint32_t* bitmask, float dropout_p, uint64_t seed,
                     void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                     void* cuda_stream);

/* The reverse pass of attn_bwd for callers that cannot allocate device memory
 * and so cannot pass a workspace: for example a plugin whose host gives it only
 * its input and output buffers, or code that must not let a device allocation
 * (which can synchronise the device or fail under a memory cap) happen on its
 * path.  This operation has no counterpart in the pages that define the
 * method; it is attn_bwd with its scratch moved into the library.
 *
 * Arguments, layouts and results are those of attn_bwd, without the workspace.
 * The scratch is a 64 MiB array in the library's own device memory, which every
 * GPU that loads this part of the library keeps until the process exits; the
 * call allocates nothing.  A problem whose exattn_bwd_workspace_size exceeds
 * 64 MiB (67108864 bytes) is rejected with EXATTN_WORKSPACE_TOO_SMALL and no
 * work is queued.  The first call on a device looks up the array's device
 * address with that device current; make that first call before any stream
 * capture.  All calls share the one array (each call clears what must start at
 * zero): calls whose work overlaps on the GPU, for example on two streams,
 * race and must not be issued.  The device status word lives in the array;
 * read it with exattn_noalloc_device_status (not exattn_device_status).
 * Returns an exattn_status. */
int attn_bwd_noalloc(const exattn_shape* shape, const void* Q, const void* K, const void* V,
                     const void* Y, const void* dY, const float* L, float scale, int mask_kind,
                     int window, const uint32_t* bitmask, void* dQ, void* dK, void* dV,
                     void* cuda_stream);

/* The device status word of the last attn_bwd_noalloc call on the current
 * device, which that call's kernels write into the library's scratch array
 * (no counterpart in the pages either).  Synchronises `cuda_stream` first (the
 * stream of that call), then reads the word.  Returns EXATTN_OK,
 * EXATTN_EMPTY_ROW (some allowed-key set was empty), EXATTN_TIMEOUT (a bounded
 * device wait gave up: the gradients are not valid) or EXATTN_CUDA_ERROR.  The
 * word is shared by every attn_bwd_noalloc call on the device and is cleared
 * at the start of each, so read it before the next call is queued. */
int exattn_noalloc_device_status(void* cuda_stream);

/* ---------------------------------------------------------------------------
 * Split-KV forward: a few queries against a long key sequence (a decode step).
 *
 * The Forward procedure of "Exact tiled softmax attention with block-
 * recomputed vector-Jacobian products" keeps a per-row summary of the key
 * blocks seen and merges it with each new block's summary (the star merge).
 * attn_fwd_splitkv cuts the keys into `num_splits` contiguous chunks handled
 * in parallel, writes every chunk's summary (running max, running sum,
 * unnormalised output) per query row to the workspace; the summaries of all
 * chunks are then merged, skipping empty ones, into Y and L (by the last CTA
 * of each slice to finish on the register kernel below, otherwise by a second
 * kernel).  The
 * result is the same attention for every num_splits (up to rounding).
 *
 * Shapes: Q [B][H][nq][d], K [B][H][nk][d], V [B][H][nk][v], Y [B][H][nq][v]
 * (dtype), L fp32 [B][H][nq] (natural log).  Query i sits at absolute position
 * i + nk - nq (the queries are the last nq positions): CAUSAL allows
 * j <= i + nk - nq, WINDOW w the w keys ending there, BITMASK reads bit rows
 * [nq][ceil(nk/32)].  Limits: 1 <= nq <= 64, nk >= 1, d, v <= 256 and rows of
 * whole 16-byte pieces (d, v multiples of 8 for bf16, of 4 for fp32),
 * 0 <= num_splits <= 4096 (chunks are whole multiples of 32 keys, of 128 for
 * the tensor-core shapes below, so fewer chunks may be used than asked for;
 * 0 picks enough chunks for about 8 waves of resident CTAs over all
 * batch*head slices, at least 256 keys each, from the shape alone, so the
 * workspace query and the call agree).  Kernels: bf16 with d = v in
 * {64, 128}, nq >= 2 and a positive scale runs the tensor-core forward in
 * summary mode per chunk, then a merge kernel; any other shape with nq <= 4
 * runs a register-resident chunk kernel that merges in its last CTA per
 * slice; the rest a shared-memory chunk kernel, then the merge kernel.  Rows with an empty
 * allowed set get Y_i = 0, L_i = -inf and the EXATTN_EMPTY_ROW status.
 * Ownership, streams and errors as for attn_fwd.
 * ------------------------------------------------------------------------- */
typedef struct exattn_qk_shape {
  int batch;
  int heads;
  int nq;
  int nk;
  int d;
  int v;
  int dtype;
} exattn_qk_shape;

/* Workspace bytes of attn_fwd_splitkv (status word, a chunk counter per slice and
 * the chunk summaries); 0 if invalid. */
size_t exattn_splitkv_workspace_size(const exattn_qk_shape* shape, int num_splits);

int attn_fwd_splitkv(const exattn_qk_shape* shape, const void* Q, const void* K, const void* V,
                     float scale, int mask_kind, int window, const uint32_t* bitmask,
                     int num_splits, void* Y, float* L, void* workspace, size_t workspace_bytes,
                     void* cuda_stream);

/* ---------------------------------------------------------------------------
 * Cross-attention: nq query rows against nk keys.
 *
 * The method of "Exact tiled softmax attention with block-recomputed vector-
 * Jacobian products" (Inputs: allowed-key sets A_i of keys per query row)
 * does not need nq == nk; "What Ordinary Autograd Saves" (The implementation
 * under test) keeps separate query and key lengths.  Here query i sits at
 * absolute position i + nk - nq (the queries are the last nq positions), so
 * CAUSAL allows j <= i + nk - nq, WINDOW w the w keys ending there, and
 * BITMASK reads bit rows [nq][ceil(nk/32)].  With nq > nk the first nq - nk
 * queries precede every key: under CAUSAL their allowed sets are empty (Y_i =
 * 0, L_i = -inf, dQ_i = 0, status EXATTN_EMPTY_ROW).
 *
 * Shapes: Q, dQ [B][H][nq][d]; K, dK [B][H][nk][d]; V, dV [B][H][nk][v];
 * Y, dY [B][H][nq][v]; L float32 [B][H][nq].  Limits as for attn_fwd, for nq
 * and nk alike.  dropout_p and seed as for attn_fwd_dropout (0: none; keep
 * decisions are indexed by the query row i and key j).  The workspace queries
 * follow attn_fwd / attn_bwd (the reverse workspace grows with nq).  With nq ==
 * nk these calls are attn_fwd_dropout / attn_bwd_dropout.  The atomic dQ form
 * does not take nq != nk: with EXATTN_PATH_ATOMIC_DQ the reverse pass of such
 * a shape runs on the SIMT kernels.
 * ------------------------------------------------------------------------- */
size_t exattn_fwd_qk_workspace_size(const exattn_qk_shape* shape, int mask_kind);
size_t exattn_bwd_qk_workspace_size(const exattn_qk_shape* shape, int mask_kind);
int attn_fwd_qk(const exattn_qk_shape* shape, const void* Q, const void* K, const void* V,
                float scale, int mask_kind, int window, const uint32_t* bitmask, float dropout_p,
                uint64_t seed, void* Y, float* L, void* workspace, size_t workspace_bytes,
                void* cuda_stream);
int attn_bwd_qk(const exattn_qk_shape* shape, const void* Q, const void* K, const void* V,
                const void* Y, const void* dY, const float* L, float scale, int mask_kind,
                int window, const uint32_t* bitmask, float dropout_p, uint64_t seed, void* dQ,
                void* dK, void* dV, void* workspace, size_t workspace_bytes, void* cuda_stream);

/* ---------------------------------------------------------------------------
 * A forward and reverse step on tensors in HOST memory: attn_fwd then
 * attn_bwd ("Exact tiled softmax attention with block-recomputed
 * vector-Jacobian products", Forward and Reverse procedures) with the copies to
 * and from the device inside the call.
 *
 * Q, K, V, dY (inputs) and Y, L, dQ, dK, dV (outputs) are host pointers with
 * the shapes and layouts of attn_fwd / attn_bwd; page-locked (pinned) memory
 * lets the copies run asynchronously and at full speed, pageable memory works
 * but the copies then block the calling thread.  `bitmask` (BITMASK only) is a
 * host pointer too.  No dropout.  `workspace` is device memory of at least
 * exattn_host_step_workspace_size bytes, 256-byte aligned: it holds device
 * copies of all nine tensors plus the working space of one chunk.
 *
 * The slices are cut into chunks (up to 8).  Chunk k's inputs are copied in on
 * one internal stream, its forward and reverse pass run on a second, and its
 * outputs are copied out on a third, so the copies of neighbouring chunks
 * overlap the kernels.  The call queues everything after the work already on
 * `cuda_stream` and returns at once; `cuda_stream` waits for the whole step,
 * so synchronising it (or exattn_device_status on `workspace`) makes the host
 * outputs valid.  Each slice's results are bitwise those of attn_fwd and
 * attn_bwd.  The status word of `workspace` is the OR over the chunks.
 * Host-side failures return before any copy is queued.  A CUDA error met while
 * queuing returns EXATTN_CUDA_ERROR (text in exattn_last_error); `cuda_stream`
 * still waits for whatever had been queued, so the buffers may be freed once it
 * is synchronised.
 * ------------------------------------------------------------------------- */
size_t exattn_host_step_workspace_size(const exattn_shape* shape, int mask_kind);
int attn_step_host(const exattn_shape* shape, const void* Q, const void* K, const void* V,
                   const void* dY, float scale, int mask_kind, int window, const uint32_t* bitmask,
                   void* Y, float* L, void* dQ, void* dK, void* dV, void* workspace,
                   size_t workspace_bytes, void* cuda_stream);

/* Waits for `cuda_stream`, then reads the status word of `workspace` (the
 * workspace of the last call queued on it).  Returns EXATTN_OK,
 * EXATTN_EMPTY_ROW, EXATTN_TIMEOUT or EXATTN_CUDA_ERROR. */
int exattn_device_status(const void* workspace, void* cuda_stream);

/* Profiling aid.  Kernels of the library, by role. */
enum exattn_kernel {
  EXATTN_KERNEL_FWD = 0,        /* the forward kernel of attn_fwd */
  EXATTN_KERNEL_DELTA = 1,      /* delta_i = dY_i . Y_i in attn_bwd (not launched on the
                                   AUTO tensor-core path: its dQ kernel forms delta) */
  EXATTN_KERNEL_BWD = 2,        /* the reverse kernel(s) of attn_bwd: start before the first,
                                   stop after the last (dQ, then dK/dV kernel on AUTO) */
  EXATTN_KERNEL_DQ_CONVERT = 3, /* fp32 dQ accumulator -> dQ (SIMT and ATOMIC_DQ paths) */
  EXATTN_KERNEL_BWD_Q = 4,      /* the query-major dQ kernel alone (AUTO path; it also
                                   forms delta_i and L_i log2 e for the dK/dV kernel) */
  EXATTN_KERNEL_SPLIT_PARTIAL = 5, /* per-chunk summaries of attn_fwd_splitkv */
  EXATTN_KERNEL_SPLIT_MERGE = 6,   /* the merge kernel of attn_fwd_splitkv (shapes
                                     whose chunks do not merge themselves) */
  EXATTN_KERNEL_SPLIT32 = 7        /* the tf32 hi / lo split of K and V (fp32 forward) */
};

/* One-shot: on the next launch of kernel `which` (an exattn_kernel), record
 * the cudaEvent_t `start` on the call's stream immediately before the launch
 * and `stop` immediately after it, then forget both.  The events are owned by
 * the caller.  Returns 0, or -1 for an unknown `which`.  Process-wide. */
int exattn_record_kernel_events(int which, void* start, void* stop);

/* Number of kernels this library has launched since it was loaded
 * (process-wide, all devices). */
unsigned long long exattn_launch_count(void);

/* Self-test of the failure path of the tensor-core kernels, whose every
 * device-side wait is bounded.  Launches one small kernel whose wait on a
 * barrier that nothing arrives on gives up after `limit_us` microseconds
 * (1..100000); it records EXATTN_TIMEOUT in the status word of `workspace`
 * (>= 256 bytes, 256-byte aligned) and returns, and a second waiter with the
 * normal 1 s limit stops early on the kernel's abort flag.  Words 1..3 of the
 * workspace receive: 1 if the first wait timed out, 1 if the second stopped on
 * the abort flag, and the second waiter's time in microseconds.  Read the
 * status with exattn_device_status (expected EXATTN_TIMEOUT).  No trap, fault
 * or unbounded wait is involved. */
int exattn_selftest_wait_timeout(void* workspace, unsigned limit_us, void* cuda_stream);

/* Text of the last CUDA failure seen by a call on this host thread (which
 * step failed and the CUDA or driver error), or "" if none.  Valid until the
 * next call on this thread. */
const char* exattn_last_error(void);

/* A static, human-readable name for a status code. */
const char* exattn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* EXATTN_H */
