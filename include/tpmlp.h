/*
 * tpmlp.h — C ABI of the GB300 (sm_103a) tensor-parallel MLP library.
 *
 * The library computes the Megatron tensor-parallel MLP
 *
 *     Y = GeLU(X A) B,     X [T, D],  A [D, F],  B [F, D],
 *
 * with A split by columns and B by the matching rows into n shards, every
 * shard's partial output computed on its own and the partials summed (the
 * simulated all-reduce). All n shards run on the one GPU that is current when
 * a call is made. Sources for each call are given beside it:
 *   [P4] scratchllm.com "Tensor-Parallel MLP (Megatron)"
 *   [P3] duoan.github.io "Tensor Parallelism in Megatron-LM"
 *   [P1] ai-hpc.org "LLM Lab Notes 06: Megatron-style Transformer Block"
 *
 * Conventions that hold for every call:
 *   - Matrices are dense and row-major (the last index is contiguous).
 *   - Pointers named as "device" point to CUDA device memory on the current
 *     device; the caller owns it unless stated otherwise. They must be 16-byte
 *     aligned (TPMLP_ERR_ALIGN otherwise).
 *   - Every call that takes a stream only enqueues work on it and returns; the
 *     results are ready when that stream has reached the point of the call.
 *     Kernels are launched with programmatic dependent launch: each one's
 *     set-up overlaps the end of the previous kernel in the stream, and it
 *     waits for that kernel to complete before it reads or writes global
 *     memory, so stream order is kept (environment variable TPMLP_PDL=0
 *     launches them plainly).
 *   - The return value is TPMLP_OK (0) or a negative tpmlp_status. On error
 *     nothing has been enqueued, and tpmlp_last_error() gives a message.
 *   - Kernels never trap. A device-side wait that runs past its time limit
 *     makes the kernel stop early and record TPMLP_ERR_TIMEOUT in a per-device
 *     status word, which tpmlp_check_status() reads and clears.
 *   - In bf16 (TPMLP_BF16) mode the operands X, A, B, dY are bf16, products are
 *     accumulated in fp32, H_i and the backward's dP_i are rounded to bf16 when
 *     they become operands of the next product, and every output (Y, dX, dA_i,
 *     dB_i) is fp32. In fp32 (TPMLP_F32) mode everything is fp32.
 */
#ifndef TPMLP_H
#define TPMLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* tpmlp_stream_t;

typedef enum { TPMLP_F32 = 0, TPMLP_BF16 = 1 } tpmlp_dtype;

/* How the shard partials are summed ([P4] "The split", third bullet).
 * FAITHFUL: every partial Y_i is written to memory, then one kernel adds them
 *           in shard order ((Y_0 + Y_1) + Y_2) + ... .
 * FUSED:    the second product walks its contraction shard by shard, 0..n-1,
 *           into one on-chip accumulator, so no partial is ever written. */
typedef enum { TPMLP_FAITHFUL = 0, TPMLP_FUSED = 1 } tpmlp_mode;

typedef enum {
  TPMLP_OK = 0,
  TPMLP_ERR_ARG = -1,          /* null pointer, non-positive size, bad enum   */
  TPMLP_ERR_DIVISIBILITY = -2, /* F not divisible by n ([P4] "What to implement") */
  TPMLP_ERR_ALIGN = -3,        /* a pointer is not 16-byte aligned            */
  TPMLP_ERR_SHAPE = -4,        /* bf16: D or F/n not a multiple of 8          */
  TPMLP_ERR_CUDA = -5,         /* a CUDA runtime call failed                  */
  TPMLP_ERR_TIMEOUT = -6,      /* a device-side wait ran out of time          */
  TPMLP_ERR_WORKSPACE = -7,    /* workspace missing or smaller than required  */
  TPMLP_ERR_UNSUPPORTED = -8,  /* e.g. bf16 with more than TPMLP_MAX_SHARDS   */
  TPMLP_ERR_DEVICE = -9,       /* current device is not sm_103 / shards handle
                                  belongs to another device                   */
  TPMLP_ERR_BOUNDS = -10       /* debug build: a device-side index check failed */
} tpmlp_status;

/* Largest shard count of the bf16 tensor-core path (the fp32 path has none). */
#define TPMLP_MAX_SHARDS 16

/* Opaque handle: the n shard pairs (A_i, B_i) and their descriptor table. */
typedef struct tpmlp_shards tpmlp_shards;

/* Library version, (major << 16) | minor. */
int tpmlp_version(void);

/* Message for the last error returned on the calling thread ("" if none). */
const char* tpmlp_last_error(void);

/* Waits for `stream`, then reads and clears the current device's status word.
 * Returns TPMLP_OK, TPMLP_ERR_TIMEOUT if a kernel gave up on a wait since the
 * last check, TPMLP_ERR_BOUNDS if a device-side check of the debug build
 * failed (see tpmlp_build_flags), or TPMLP_ERR_CUDA if the stream reports an
 * error or a kernel found its dynamic shared memory misaligned (it then did
 * no work). The first failure since the last check is the one reported. */
int tpmlp_check_status(tpmlp_stream_t stream);

/* Build flags of the loaded library: bit 0 is set in the debug build
 * (compiled with TPMLP_DEBUG; the Python binding loads it as
 * libtpmlp_debug.so when TPMLP_DEBUG=1 is set). In that build the kernels
 * check their tile, TMA-coordinate, output, reduce-slice and attention-tile
 * indices on the device; a failed check skips the access it guards (the
 * kernel does not trap), stops the kernel's work where skipping would leave
 * it waiting, and records TPMLP_ERR_BOUNDS for tpmlp_check_status. The
 * results of the two builds are identical when no check fails. */
int tpmlp_build_flags(void);

/* Test hook for the debug build's checks: one block writes element `index`
 * of a 32-element shared-memory array, guarded by a device-side check. With
 * 0 <= index < 32 nothing is recorded; otherwise the check fails, the write
 * is skipped and the next tpmlp_check_status() returns TPMLP_ERR_BOUNDS.
 * Returns TPMLP_ERR_UNSUPPORTED (and launches nothing) in the normal build. */
int tpmlp_selftest_bounds(int index, tpmlp_stream_t stream);

/* gelu(x), elementwise: GeLU(x) = 1/2 x (1 + tanh u), u = sqrt(2/pi)(x + 0.044715 x^3)
 * ([P4] section "GeLU"; "What to implement", first bullet).
 *   x, y  device arrays of n elements of type dt (y may equal x).
 *   n     element count, >= 0 (0 enqueues nothing).
 * Computed in fp32; the bf16 variant rounds the result once to bf16. */
int tpmlp_gelu(const void* x, void* y, int64_t n, tpmlp_dtype dt, tpmlp_stream_t stream);

/* shard_mlp(A, B, n): split A [D, F] by columns and B [F, D] by rows into n
 * pairs; shard i receives columns i*F/n .. (i+1)*F/n - 1 of A and the same
 * rows of B ([P4] "What to implement", second bullet, and "Requirements").
 *   A, B   device, row-major, of type dt; only read (the copies are enqueued
 *          on `stream`, so A and B must stay valid until it reaches them).
 *   n      1 <= n; F % n == 0 (TPMLP_ERR_DIVISIBILITY); bf16 needs n <=
 *          TPMLP_MAX_SHARDS and D, F/n multiples of 8 (TPMLP_ERR_SHAPE).
 *   out    receives the handle. The handle owns device copies of every A_i and
 *          B_i (and, for bf16, their transposes, the operand layouts of the
 *          tensor-core kernels) plus the device descriptor table, all made
 *          with cudaMalloc on the current device; release them with
 *          tpmlp_shards_free(). */
int tpmlp_shard(const void* A, const void* B, int64_t D, int64_t F, int n, tpmlp_dtype dt,
                tpmlp_stream_t stream, tpmlp_shards** out);

/* Shape of a handle. Any output pointer may be NULL. */
int tpmlp_shard_info(const tpmlp_shards* shards, int64_t* D, int64_t* F, int* n, tpmlp_dtype* dt);

/* Device pointers to shard i's A_i [D, F/n] and B_i [F/n, D] (row-major,
 * owned by the handle, valid until tpmlp_shards_free). */
int tpmlp_shard_get(const tpmlp_shards* shards, int i, const void** A_i, const void** B_i);

/* bf16 handles only: shard i's transposed copies A_i^T [F/n, D] and
 * B_i^T [D, F/n] (row-major, owned by the handle). TPMLP_ERR_UNSUPPORTED for
 * fp32 handles, which keep no transposes. */
int tpmlp_shard_get_transposed(const tpmlp_shards* shards, int i, const void** At_i, const void** Bt_i);

/* Releases everything the handle owns (synchronises the device first). NULL is a no-op. */
void tpmlp_shards_free(tpmlp_shards* shards);

/* Bytes of workspace that tpmlp_forward / tpmlp_forward_save (backward = 0),
 * tpmlp_backward (backward = 1) or tpmlp_backward_saved (backward = 2) needs
 * for T tokens, these shards and this mode; 0 on bad arguments. The workspace
 * holds the shards' H_i (and, in FAITHFUL mode, the partials), so it grows
 * with T * F and, for FAITHFUL, with n * T * D. */
size_t tpmlp_workspace_bytes(int64_t T, const tpmlp_shards* shards, tpmlp_mode mode, int backward);

/* tp_mlp(X, shards): Y = sum_i GeLU(X A_i) B_i ([P4] "What to implement",
 * third bullet; [P3] §3 "The MLP Block").
 *   X    device [T, D] of the handle's dtype.
 *   T    >= 1 tokens.
 *   Y    device [T, D] fp32, written (not accumulated).
 *   workspace, workspace_bytes  device scratch of at least
 *        tpmlp_workspace_bytes(T, shards, mode, 0) bytes, caller-owned; its
 *        contents are undefined afterwards.
 * FAITHFUL sums the partials in shard order and is bitwise reproducible from
 * run to run; FUSED gives the same sum to within rounding. */
int tpmlp_forward(const void* X, int64_t T, const tpmlp_shards* shards, void* Y, tpmlp_mode mode,
                  void* workspace, size_t workspace_bytes, tpmlp_stream_t stream);

/* The steps of tpmlp_forward, one call each, for callers that keep the
 * intermediates.
 *
 * tpmlp_hidden: H_i = GeLU(X A_i) for every shard i ([P4] "The split", first
 * bullet; [P3] §3 steps 1-2). X device [T, D]; H device [n][T][F/n] of the
 * handle's dtype (shard i's block starts at H + i*T*(F/n) elements). */
int tpmlp_hidden(const void* X, int64_t T, const tpmlp_shards* shards, void* H, tpmlp_stream_t stream);

/* tpmlp_partials: Y_i = H_i B_i for every shard i ([P4] "The split", second
 * bullet; [P3] §3 step 3). H as written by tpmlp_hidden; Yp device
 * [n][T][D] fp32 (shard i's partial starts at Yp + i*T*D). */
int tpmlp_partials(const void* H, int64_t T, const tpmlp_shards* shards, void* Yp, tpmlp_stream_t stream);

/* tpmlp_allreduce: the simulated all-reduce Y = ((Y_0 + Y_1) + ...) + Y_{n-1}
 * in fp32, in shard order ([P4] "The split", third bullet; [P1] §2 note 6).
 * Yp device [n][count] fp32; Y device [count] fp32 (must not overlap Yp). */
int tpmlp_allreduce(const void* Yp, int n, int64_t count, void* Y, tpmlp_stream_t stream);

/* tpmlp_fused_sum: Y = sum_i H_i B_i accumulated shard by shard (0..n-1) on
 * chip, with no partial written ([P3] §3: reduce where partial linear
 * outputs must be summed). H as written by tpmlp_hidden; Y device [T, D] fp32. */
int tpmlp_fused_sum(const void* H, int64_t T, const tpmlp_shards* shards, void* Y, tpmlp_stream_t stream);

/* Backward of Y = sum_i GeLU(X A_i) B_i for the upstream gradient dY, i.e. the
 * gradients of L = sum(Y * dY) ([P3] §3, the f/g operators; [P1] §2 note 8):
 *   P_i = X A_i (recomputed), dH_i = dY B_i^T, dP_i = dH_i * GeLU'(P_i),
 *   dB_i = H_i^T dY, dA_i = X^T dP_i, dX = sum_i dP_i A_i^T (shard order in
 *   FAITHFUL mode, on-chip accumulation in FUSED mode).
 * dY reaches every shard unchanged; only dX is summed over shards.
 *   X, dY  device [T, D] of the handle's dtype.
 *   dX     device [T, D] fp32.
 *   dA     host array of n device pointers, dA[i] -> fp32 [D, F/n].
 *   dB     host array of n device pointers, dB[i] -> fp32 [F/n, D].
 *   workspace  at least tpmlp_workspace_bytes(T, shards, mode, 1) bytes. */
int tpmlp_backward(const void* X, const void* dY, int64_t T, const tpmlp_shards* shards, void* dX,
                   void* const* dA, void* const* dB, tpmlp_mode mode, void* workspace,
                   size_t workspace_bytes, tpmlp_stream_t stream);

/* Test hook for the time limits inside the tensor-core product: runs the
 * H_i = GeLU(X A_i) product of tpmlp_hidden (bf16 shards only) with stage
 * fill number `fill` (1-based, counted by each CTA's producer) never issued,
 * and a wait limit of limit_ms (1..10000). Every CTA that reaches that fill
 * gives up after the limit, drains its copies and MMAs, frees its tensor
 * memory and records TPMLP_ERR_TIMEOUT, which the next tpmlp_check_status()
 * returns; the other CTAs finish normally. H is left partly written.
 * TPMLP_ERR_UNSUPPORTED for fp32 shards. */
int tpmlp_selftest_gemm_withheld_fill(const void* X, int64_t T, const tpmlp_shards* shards, void* H, int fill,
                                      int limit_ms, tpmlp_stream_t stream);

/* Test hook for the persistent forward's band waits (the one-launch form that
 * tpmlp_forward takes for small and mid-size bf16 products whose weights fit
 * in L2): runs it with every band of H
 * needing one arrival more than its first-product tiles make, so the
 * producer of every second-product tile waits for a band that is never
 * complete and gives up after limit_ms (1..10000); the kernel drains its
 * copies and products, frees its tensor memory and records TPMLP_ERR_TIMEOUT
 * for the next tpmlp_check_status(). Y (and, FAITHFUL, the workspace's
 * partials) are left partly written; no reduce runs. Arguments as
 * tpmlp_forward; TPMLP_ERR_UNSUPPORTED if this forward would not run as one
 * launch. */
int tpmlp_selftest_forward_band_timeout(const void* X, int64_t T, const tpmlp_shards* shards, void* Y, tpmlp_mode mode,
                                        void* workspace, size_t ws_bytes, int limit_ms, tpmlp_stream_t stream);

/* Test hook for the recomputing backward's first step (the dual-accumulator
 * kernel, used for bf16 products with enough CTA-pair tiles): runs that
 * kernel alone with stage fill number `fill` (1-based, counted by each CTA's
 * producer) never issued and a wait limit of limit_ms (1..10000). Every CTA
 * pair that reaches the fill gives up, drains, frees its tensor memory and
 * records TPMLP_ERR_TIMEOUT. Workspace as tpmlp_backward in FUSED mode (its
 * H and dP parts are left partly written). TPMLP_ERR_UNSUPPORTED if this
 * backward would not use the dual kernel. */
int tpmlp_selftest_backward_withheld_fill(const void* X, const void* dY, int64_t T, const tpmlp_shards* shards,
                                          int fill, int limit_ms, void* workspace, size_t ws_bytes,
                                          tpmlp_stream_t stream);

/* tpmlp_forward without any allocation: the same Y, but the scratch lives in
 * a fixed 64 MiB array of device memory that the library reserves on every
 * GPU where its device code is loaded and keeps until the process exits. (The
 * pages have no counterpart to this call; it exists for the library's users.)
 * For callers that cannot allocate device memory at call time — runtimes that
 * own all GPU memory through their own pool and forbid allocations outside
 * it, or loops that cannot take the device synchronisation of cudaMalloc /
 * cudaFree — and so cannot pass the workspace tpmlp_forward needs.
 *   X, T, shards, Y, mode, stream  as for tpmlp_forward.
 * Allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 * TPMLP_ERR_WORKSPACE if tpmlp_workspace_bytes(T, shards, mode, 0) exceeds
 * 64 MiB (at D=4096, F=16384, n=8: above 2048 tokens in FUSED mode, above
 * 409 tokens in FAITHFUL mode).
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture. All calls on a GPU share the one array, so calls whose work
 * may overlap on the GPU race on it; order them on one stream. Nothing in the
 * array needs to start at zero, and it keeps the last call's contents. */
int tpmlp_forward_noalloc(const void* X, int64_t T, const tpmlp_shards* shards, void* Y, tpmlp_mode mode,
                          tpmlp_stream_t stream);

/* Training-mode forward: the same Y as tpmlp_forward, and in addition the
 * shards' pre-activations P_i = X A_i (fp32), which tpmlp_backward_saved
 * uses instead of recomputing them. ai-hpc.org "LLM Lab Notes 06" §4 notes
 * that the backward costs about the sum of the forward passes; keeping P
 * removes the recompute (2*T*D*F of the backward's 10*T*D*F FLOP) at the
 * price of T*F*4 bytes.
 *   P     device [n][T][F/n] fp32, written (shard i's block at P + i*T*(F/n)).
 *   other arguments as for tpmlp_forward (same workspace size). */
int tpmlp_forward_save(const void* X, int64_t T, const tpmlp_shards* shards, void* Y, void* P, tpmlp_mode mode,
                       void* workspace, size_t workspace_bytes, tpmlp_stream_t stream);

/* tpmlp_backward with the P written by tpmlp_forward_save for the same X and
 * shards: the same dX, dA_i, dB_i without recomputing P (P is only read).
 *   workspace  at least tpmlp_workspace_bytes(T, shards, mode, 2) bytes. */
int tpmlp_backward_saved(const void* X, const void* dY, const void* P, int64_t T, const tpmlp_shards* shards,
                         void* dX, void* const* dA, void* const* dB, tpmlp_mode mode, void* workspace,
                         size_t workspace_bytes, tpmlp_stream_t stream);

/* ------------------------------------------------------------------------
 * The FFN half of a transformer block ([P1] §2 steps 5-7 and 8):
 *
 *     out = x + sum_i GeLU(LN(x) A_i) B_i,
 *
 * LN the row-wise layer norm (x - mean) / sqrt(var + eps) with the biased
 * variance and no scale or shift ([P1] calls it with the hidden size only).
 * The residual x is added to the finished shard sum ([P1] §2: the all-reduced
 * output, then the residual). In bf16 mode LN(x) is rounded to bf16 when it
 * becomes the first product's operand, like every other operand.
 * ---------------------------------------------------------------------- */

/* y = LN(x) row by row. x, y device [T, D] of type dt (may be the same
 * buffer); T >= 0, 1 <= D <= 25536 (TPMLP_ERR_SHAPE above); eps > 0 and
 * finite. Statistics in fp32, two-pass (mean, then mean squared deviation). */
int tpmlp_layer_norm(const void* x, int64_t T, int64_t D, tpmlp_dtype dt, float eps, void* y, tpmlp_stream_t stream);

/* Workspace bytes tpmlp_block_forward (backward = 0) or tpmlp_block_backward
 * (backward = 1) needs; 0 on bad arguments. */
size_t tpmlp_block_workspace_bytes(int64_t T, const tpmlp_shards* shards, tpmlp_mode mode, int backward);

/* out = x + sum_i GeLU(LN(x) A_i) B_i.
 *   x    device [T, D] of the handle's dtype: the block input and residual.
 *   eps  the layer norm's eps (PyTorch's default is 1e-5).
 *   out  device [T, D] fp32, written; must not overlap x.
 *   xn   device [T, D] of the handle's dtype that receives LN(x) as it entered
 *        the first product, or NULL (then it lives in the workspace).
 *   mode FAITHFUL: shard partials, then one pass that sums them in shard
 *        order and adds x (out = x + (((Y_0 + Y_1) + ...))); FUSED: on-chip
 *        shard-ordered accumulation with x added in the product's epilogue.
 *   workspace  at least tpmlp_block_workspace_bytes(T, shards, mode, 0). */
int tpmlp_block_forward(const void* x, int64_t T, const tpmlp_shards* shards, float eps, void* out, void* xn,
                        tpmlp_mode mode, void* workspace, size_t workspace_bytes, tpmlp_stream_t stream);

/* Backward of tpmlp_block_forward for the upstream gradient dout: the
 * gradients of L = sum(out * dout) ([P1] §2 step 8). The residual passes dout
 * to x; the MLP's backward (as in tpmlp_backward, with X = LN(x) recomputed
 * and dY = dout) gives dA_i, dB_i and the gradient g of LN(x), which goes back
 * through the norm:
 *   dx = dout + r (g - mean(g) - y mean(g * y)),  y = LN(x), r = 1/sqrt(var + eps),
 * with g the shard-ordered sum of the partials in FAITHFUL mode (summed in the
 * same pass) and the on-chip sum in FUSED mode.
 *   x, dout  device [T, D] of the handle's dtype.
 *   dx       device [T, D] fp32.
 *   dA, dB   as for tpmlp_backward.
 *   workspace  at least tpmlp_block_workspace_bytes(T, shards, mode, 1). */
int tpmlp_block_backward(const void* x, const void* dout, int64_t T, const tpmlp_shards* shards, float eps, void* dx,
                         void* const* dA, void* const* dB, tpmlp_mode mode, void* workspace,
                         size_t workspace_bytes, tpmlp_stream_t stream);

/* ------------------------------------------------------------------------
 * Sequence-parallel form ([P3] "Row split": the partials are summed by an
 * all-reduce, or by reduce-scatter / all-gather when the sequence is split).
 * The n ranks are the n shards; T must be divisible by n, and rank j holds
 * token rows j*T/n .. (j+1)*T/n - 1 of X (and dY) and receives the same rows
 * of the output (and of dX). Each call takes host arrays of n device
 * pointers, one per rank slice, each 16-byte aligned. n <= TPMLP_MAX_SHARDS
 * (TPMLP_ERR_UNSUPPORTED above), T % n != 0 gives TPMLP_ERR_DIVISIBILITY.
 * ---------------------------------------------------------------------- */

/* The simulated all-gather: out = slices[0] .. slices[n-1] back to back,
 * slice_bytes (a multiple of 2) each. out device, n * slice_bytes bytes,
 * overlapping no slice. */
int tpmlp_all_gather(const void* const* slices, int n, int64_t slice_bytes, void* out, tpmlp_stream_t stream);

/* The simulated reduce-scatter: the shard-ordered fp32 sum
 * ((Yp_0 + Yp_1) + ...) + Yp_{n-1} of the partials Yp device [n][count]
 * fp32, cut into n equal slices; slice j (count/n elements, count % n == 0)
 * goes to Y_slices[j] (device fp32). Bit-identical to the matching part of
 * tpmlp_allreduce. */
int tpmlp_reduce_scatter(const void* Yp, int n, int64_t count, void* const* Y_slices, tpmlp_stream_t stream);

/* Workspace bytes tpmlp_forward_sp (backward = 0) or tpmlp_backward_sp
 * (backward = 1) needs; 0 on bad arguments (incl. T % n != 0). */
size_t tpmlp_sp_workspace_bytes(int64_t T, const tpmlp_shards* shards, tpmlp_mode mode, int backward);

/* Sequence-parallel forward: X = all-gather of the n slices, every shard's
 * partial of GeLU(X A_i) B_i, and rank j's rows of the shard-ordered sum
 * written to Y_slices[j].
 *   X_slices  n device pointers, [T/n, D] of the handle's dtype.
 *   Y_slices  n device pointers, [T/n, D] fp32.
 *   mode      FAITHFUL: partials, then the reduce-scatter kernel; FUSED: the
 *             on-chip shard-ordered sum, whose epilogue writes each output
 *             row straight into its rank's slice.
 *   workspace at least tpmlp_sp_workspace_bytes(T, shards, mode, 0). */
int tpmlp_forward_sp(const void* const* X_slices, int64_t T, const tpmlp_shards* shards, void* const* Y_slices,
                     tpmlp_mode mode, void* workspace, size_t workspace_bytes, tpmlp_stream_t stream);

/* Sequence-parallel backward: X and dY all-gathered from their slices, the
 * gradients of tpmlp_backward, and dX reduce-scattered: rank j's rows of
 * dX = sum_i dP_i A_i^T go to dX_slices[j] ([T/n, D] fp32). dA, dB as for
 * tpmlp_backward (every rank's shard gradient is whole).
 *   workspace at least tpmlp_sp_workspace_bytes(T, shards, mode, 1). */
int tpmlp_backward_sp(const void* const* X_slices, const void* const* dY_slices, int64_t T,
                      const tpmlp_shards* shards, void* const* dX_slices, void* const* dA, void* const* dB,
                      tpmlp_mode mode, void* workspace, size_t workspace_bytes, tpmlp_stream_t stream);

/* ------------------------------------------------------------------------
 * Head-split attention ([P3] §4 "Attention: Split Heads"; [P1] §2 steps 2-3):
 * H heads of size d_h = D / H; rank i owns heads i*H/n .. (i+1)*H/n - 1,
 * i.e. columns i*D/n .. (i+1)*D/n - 1 of Wq, Wk, Wv [D, D] (column-parallel)
 * and the same rows of Wo [D, D] (row-parallel). X [T, D] holds `batch`
 * sequences of `seq` tokens (sequence b in rows b*seq .. (b+1)*seq - 1):
 *   Q_i = X Wq_i, K_i = X Wk_i, V_i = X Wv_i,
 *   O_i = softmax(Q_i K_i^T / sqrt(d_h)) V_i per sequence and local head
 *         (no mask),
 *   Y   = sum_i O_i Wo_i, summed like the MLP's partials.
 * bf16: d_h = 64, seq % 8 == 0, any length (a streaming kernel with a running
 * maximum; environment variable TPMLP_ATTN_KERNEL=0 selects, up to 512
 * tokens, an exact kernel that holds the whole score row); fp32: d_h <= 128,
 * seq <= 8192.
 * ---------------------------------------------------------------------- */

typedef struct tpmlp_attn_shards tpmlp_attn_shards;

/* Builds the ranks' weights on the current device (enqueued on `stream`).
 *   Wq, Wk, Wv, Wo  device [D, D] of type dt, read only.
 *   heads           H; D % H == 0 and H % n == 0 (TPMLP_ERR_DIVISIBILITY).
 *   n               1 .. TPMLP_MAX_SHARDS ranks.
 * Layout per rank, bf16: [Wq_i | Wk_i | Wv_i]^T [3D/n, D] and Wo_i^T
 * [D, D/n] (K-major operands of the tensor cores); fp32: [Wq_i | Wk_i | Wv_i]
 * [D, 3D/n] and Wo_i [D/n, D]. TPMLP_ERR_UNSUPPORTED for a bf16 head size
 * other than 64 or an fp32 head size above 128. */
int tpmlp_attn_shard(const void* Wq, const void* Wk, const void* Wv, const void* Wo, int64_t D, int heads, int n,
                     tpmlp_dtype dt, tpmlp_stream_t stream, tpmlp_attn_shards** out);

/* Rank i's two weight blocks in the layout above (owned by the handle). */
int tpmlp_attn_shard_get(const tpmlp_attn_shards* shards, int i, const void** Wqkv_i, const void** Wo_i);

/* Synchronises the handle's device and frees the handle (NULL is a no-op). */
void tpmlp_attn_shards_free(tpmlp_attn_shards* shards);

/* Workspace bytes of tpmlp_attn_forward in `mode` (TPMLP_FAITHFUL or
 * TPMLP_FUSED), or of tpmlp_attn_heads for mode = -1; 0 on bad arguments. */
size_t tpmlp_attn_workspace_bytes(int64_t batch, int64_t seq, const tpmlp_attn_shards* shards, int mode);

/* Every rank's local heads: O device [n][T][D/n] of the handle's dtype, rank
 * i's block at O + i*T*D/n, head h of the rank in its columns h*d_h ..
 * (h+1)*d_h - 1. workspace: tpmlp_attn_workspace_bytes(batch, seq, shards, -1). */
int tpmlp_attn_heads(const void* X, int64_t batch, int64_t seq, const tpmlp_attn_shards* shards, void* O,
                     void* workspace, size_t workspace_bytes, tpmlp_stream_t stream);

/* Y = sum_i O_i Wo_i, device [T, D] fp32. FAITHFUL: the partials O_i Wo_i,
 * then the shard-ordered reduce of tpmlp_allreduce; FUSED: their on-chip
 * shard-ordered sum. workspace: tpmlp_attn_workspace_bytes(batch, seq,
 * shards, mode). */
int tpmlp_attn_forward(const void* X, int64_t batch, int64_t seq, const tpmlp_attn_shards* shards, void* Y,
                       tpmlp_mode mode, void* workspace, size_t workspace_bytes, tpmlp_stream_t stream);

/* Per-step timing, switched on by TPMLP_TRACE=1 in the environment (read once
 * per process; the method the pages use to find where a layer's time goes,
 * [P1] section 5, "profile in segments"). While it is on, every step of a call
 * that launches device work (gemm1_gelu, gemm2_partials, allreduce,
 * gemm2_fused_sum, bwd_dual_P_dH, bwd_dB, bwd_dA, bwd_dX_partials, layer_norm,
 * attn_core, ...) is bracketed by two CUDA events on the call's stream. Steps
 * enqueued on a stream that is capturing a CUDA graph are not recorded.
 * tpmlp_trace_read waits for every recorded step to finish, then writes one
 * line per step, "<name> <milliseconds>\n", in the order the steps were
 * enqueued (across all threads), into buf (bytes long, NUL-terminated), sets
 * *records (may be NULL) to the number of lines written and forgets the
 * steps. Returns TPMLP_OK; TPMLP_ERR_WORKSPACE if buf could not hold every
 * line (the rest are dropped) or if more than 65536 steps were enqueued since
 * the last read; TPMLP_ERR_ARG if buf is NULL while bytes > 0. With tracing off
 * it writes an empty string. tpmlp_trace_enabled returns 1 if tracing is on. */
int tpmlp_trace_read(char* buf, size_t bytes, int* records);
int tpmlp_trace_enabled(void);

/* Test hook for the time limits: launches one block that waits on a device
 * barrier nobody ever completes, with the library's bounded wait and a limit
 * of limit_ms milliseconds (1..10000). The block then stops and records
 * TPMLP_ERR_TIMEOUT, which the next tpmlp_check_status() returns. */
int tpmlp_selftest_wait_timeout(int limit_ms, tpmlp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TPMLP_H */
