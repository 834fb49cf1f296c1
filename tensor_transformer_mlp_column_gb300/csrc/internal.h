// internal.h — declarations shared by the library's translation units
// (kernel launchers and the tensor-map helper). Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tpmlp {

constexpr int kMaxGroups = 16;  // shards per tensor-core launch (TPMLP_MAX_SHARDS)

// Status codes of the device-side checks (stored in the device status word):
// the bounded waits, and the shared-memory alignment check.
enum WaitSite : int {
  kSiteProducer = 1,
  kSiteMmaFull = 2,
  kSiteMmaAcc = 3,
  kSiteEpilogue = 4,
  kSiteSelftest = 5,
  kSiteSmemAlign = 6,  // a kernel found its dynamic shared memory misaligned and returned without work
  kSiteBand = 7,       // the persistent forward: a band of H was not complete in time
  kSiteBoundsBase = 16,  // debug build: a device-side check (DebugCheck) failed; the word holds 16 + the check
};

// Device-side checks of the debug build (TPMLP_DCHECK in device.cuh).
enum DebugCheck : int {
  kChkTile = 1,      // a GEMM tile index decoded outside the tile grid or the group count
  kChkTmaX = 2,      // a TMA load's inner coordinate not on a 16-byte boundary
  kChkOutput = 3,    // an epilogue store outside the output
  kChkReduce = 4,    // a reduce / gather index outside its slice
  kChkAttnTile = 5,  // an attention query tile, head or sequence outside the launch's bounds
  kChkSelftest = 6,  // tpmlp_selftest_bounds: the requested index is outside its 32-element array
  kChkCount = 7,
};

// Whether this library was built with the device-side checks (TPMLP_DEBUG).
constexpr bool kDebugBuild =
#ifdef TPMLP_DEBUG
    true;
#else
    false;
#endif

// Output treatment of the tensor-core GEMM.
enum TcEpilogue : int {
  kEpiGeluBf16 = 0,  // out bf16 = GeLU(acc)
  kEpiF32 = 1,       // out fp32 = acc
  kEpiBwdAct = 2,    // acc = dH: out bf16 = dH * GeLU'(P), out2 bf16 = GeLU(P) (P from aux_p), row-major
  kEpiF32Tma = 3,    // out fp32 = acc through TMA stores (chosen by the launcher when map_out is given)
  kEpiGeluSaveP = 4, // out bf16 = GeLU(acc) and out2 fp32 = acc (the pre-activation), same row stride
  kEpiBf16 = 5,      // out bf16 = acc
  kEpiGeluTma = 6,   // out bf16 = GeLU(acc) through TMA stores (chosen by the launcher when map_out is given)
};

enum TcShared : int { kSharedNone = 0, kSharedA = 1, kSharedB = 2 };

// One grouped GEMM on the tensor cores: for every group g,
//   out[g][m, n] = sum_k Aop_g[m, k] * Bop_g[n, k]        (chain == 0)
// or, with chain == 1, a single output
//   out[0][m, n] = sum_g sum_k Aop_g[m, k] * Bop_g[n, k]  (groups in order 0..G-1).
// Both operands are bf16, K-major (row-major with K contiguous) unless
// mn_major says otherwise, described by 2-D TMA maps made with
// make_operand_map().
struct TcGemm {
  const CUtensorMap* map_a[kMaxGroups];  // M x K operand of each group
  const CUtensorMap* map_b[kMaxGroups];  // N x K operand of each group
  const CUtensorMap* map_b_narrow[kMaxGroups];  // optional: the same operands in 64-row boxes (narrow single-CTA
                                                // tiles; used only when every group has one)
  void* out[kMaxGroups];                 // row-major outputs, row stride ldo
  void* out2[kMaxGroups];                // kEpiGeluSaveP: fp32 pre-activation; kEpiBwdAct: H (bf16); row stride ldo
  const CUtensorMap* map_out[kMaxGroups];  // optional output maps for TMA stores (fp32: make_output_map_f32; GeLU: _bf16)
  const void* aux_p[kMaxGroups];         // kEpiBwdAct only: P (fp32, row stride ldo)
  void* aux_ht[kMaxGroups];              // kEpiBf16 only: V^T (bf16, row stride ldt)
  int64_t ldo;
  int64_t ldt;
  int M, N, K;
  int groups;
  int chain;
  int epi;     // TcEpilogue
  int inject;  // test hook, 0 = off
  int shared;      // TcShared: an operand read by every group (tile order exploits it)
  int group_m;     // tile rows per band of the tile order (see decode_tile); 0 or 1 = columns fastest
  int stream_out;  // 1: evict-first epilogue stores
  const void* resid;  // kEpiF32 (and its TMA-store form): bf16 residual [M][ldo] added to acc, or null
  int64_t slice_rows;  // chain == 1, kEpiF32: rows m go to out[m / slice_rows] (with output maps, one map per
                       // slice of slice_rows rows); 0 = off
  int vt_col0;         // kEpiBf16 with aux_ht[g]: output columns >= vt_col0 are written transposed to aux_ht[g]
                       // (bf16, row pitch ldt) instead of to out[g]
  int mn_major;        // TcMajor bits: kMnA: map_a holds the M x K operand MN-major, i.e. a row-major [K][M]
                       // tensor (M contiguous), either as a 2-D map in 64 x 64 boxes (make_operand_map with
                       // 64-row boxes) or, with kMnA3d, as a 3-D map (make_operand_map_mn3d); kMnB, kMnB3d: the
                       // same for map_b and the N x K operand
};

enum TcMajor : int { kMnA = 1, kMnB = 2, kMnA3d = 4, kMnB3d = 8 };

// The backward's first step for every shard i in one kernel (gemm_dual.cu):
// P_i = X A_i and dH_i = dY B_i^T accumulated in tensor memory, then
// h[i] = GeLU(P_i) and dp[i] = dH_i * GeLU'(P_i), bf16 [M][ldo]. All four
// operand maps are K-major with 128-row boxes: X, dY [M][K]; A_i^T, B_i [N][K].
struct DualBwd {
  const CUtensorMap* map_x;
  const CUtensorMap* map_dy;
  const CUtensorMap* map_at[kMaxGroups];
  const CUtensorMap* map_b[kMaxGroups];
  void* h[kMaxGroups];
  void* dp[kMaxGroups];
  int64_t ldo;
  int M, N, K;
  int groups;
  int group_m;    // tile order (decode_tile), X and dY shared by every group
  int load_hint;  // L2 policy kinds of the M x K loads (bits 0-1) and the N x K loads (2-3)
  int inject;     // test hook: > 0 withholds that stage fill (1-based) in every CTA
};
cudaError_t launch_dual_bwd(const DualBwd& d, uint64_t wait_ns, cudaStream_t s);

// The bf16 forward's two products in one persistent launch of CTA pairs
// (gemm_fwd.cu): h[i] = GeLU(X A_i), then Y = sum_i H_i B_i (chain) or the
// partials Y_i = H_i B_i, second-product tiles starting as soon as their band
// of 256 rows of every H_i is written. Maps: X [M][K1], A_i^T [N1][K1], H_i
// [M][N1] and B_i^T [N2][N1], all K-major with 128-row boxes; map_out the fp32
// output(s) in 32 x 32 boxes (one with chain, else one per shard). band_done:
// ceil(M / 256) ints of scratch, zeroed by the launch itself.
struct FwdPersistent {
  const CUtensorMap* map_x;
  const CUtensorMap* map_at[kMaxGroups];
  const CUtensorMap* map_h[kMaxGroups];
  const CUtensorMap* map_bt[kMaxGroups];
  const CUtensorMap* map_bt64[kMaxGroups];  // B_i^T in 64-row boxes
  const CUtensorMap* map_out[kMaxGroups];
  void* h[kMaxGroups];
  int M, N1, N2, K1;
  int groups, chain;
  int* band_done;
  int band_extra;  // test hook: arrivals a band needs beyond its epilogue warps' (> 0: never complete)
};
cudaError_t launch_fwd_persistent(const FwdPersistent& f, uint64_t wait_ns, cudaStream_t s);
// CTA pairs of the persistent forward that fit the device at once (0 if it
// cannot be launched).
int fwd_persistent_clusters();
// Width of the persistent forward's second-product tiles: 128 for a
// shard-ordered sum (chain) whose 256 x 256 tiles number at most half the CTA
// pairs (twice the tiles, each half as long), else 256
// (TPMLP_FWD_NARROW2=0: always 256).
int fwd_second_width(int64_t M, int64_t N2, int chain);

// Encodes a TMA map for a row-major bf16 matrix [rows, cols] with row pitch
// `pitch_elems` (cols contiguous), boxes of 64 columns x box_rows rows and
// 128-byte swizzling. Returns false if the driver rejects it.
bool make_operand_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t pitch_elems,
                      int box_rows);

// Encodes a 3-D TMA map of a row-major bf16 matrix [rows, cols] (row pitch
// pitch_elems) read as an MN-major operand: cols / 64 chunks of 64 columns,
// each box two chunks x 64 rows (16 KB, one instruction where the 2-D map
// takes two). Needs cols % 64 == 0; returns false otherwise or if the driver
// rejects it.
bool make_operand_map_mn3d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t pitch_elems);

// Encodes a TMA map for an fp32 output matrix [rows, cols] (row pitch
// pitch_elems) written in 32 x 32 boxes with 128-byte swizzling.
bool make_output_map_f32(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t pitch_elems);
// The same for a bf16 output matrix, written in 64-column x 32-row boxes.
bool make_output_map_bf16(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t pitch_elems);
// Box heights of the two operands used by the tensor-core kernel.
int tc_box_rows_a();       // M x K operand (rows of the output)
int tc_box_rows_b(int N);  // N x K operand of a product with N output columns

cudaError_t launch_tc_gemm(const TcGemm& g, uint64_t wait_ns, cudaStream_t s);
// Whether products with enough 256 x 256 tiles run on CTA pairs (the default;
// TPMLP_TC_KERNEL=0 keeps every product on single CTAs).
bool tc_pairs_enabled();

// fp32 CUDA-core GEMM with arbitrary element strides:
//   C[m, n] (op)= sum_k A[m*sam + k*sak] * B[k*sbk + n*sbn]
enum SimtEpilogue : int { kSimtStore = 0, kSimtGelu = 1, kSimtAccumulate = 2 };
struct SimtGemm {
  const float* A;
  int64_t sam, sak;
  const float* B;
  int64_t sbk, sbn;
  float* C;
  int64_t ldc;
  int M, N, K;
  int epi;
};
cudaError_t launch_simt_gemm(const SimtGemm& g, cudaStream_t s);

cudaError_t launch_gelu(const void* x, void* y, int64_t n, int is_bf16, cudaStream_t s);
// Pointer tables passed by value to the collective kernels (one per rank slice).
struct OutSlices {
  float* p[kMaxGroups];
};
struct InSlices {
  const void* p[kMaxGroups];
};

// Y = ((Yp[0] + Yp[1]) + ...) + Yp[n-1], and with a residual res (res_kind 1:
// fp32, 2: bf16) Y = res + that sum.
cudaError_t launch_allreduce(const float* Yp, int n, int64_t count, float* Y, cudaStream_t s,
                             const void* res = nullptr, int res_kind = 0);
// The same sum cut into nslices equal slices of count / nslices elements, slice
// j written to out.p[j] (the simulated reduce-scatter; nslices = 1 is the
// all-reduce).
cudaError_t launch_reduce_scatter(const float* Yp, int n, int64_t count, const OutSlices& out, int nslices,
                                  cudaStream_t s, const void* res = nullptr, int res_kind = 0);
// out = in.p[0] .. in.p[nslices-1] back to back, slice_bytes each (a multiple
// of 2; the simulated all-gather).
cudaError_t launch_all_gather(const InSlices& in, int nslices, int64_t slice_bytes, void* out, cudaStream_t s);

// Row-wise layer norm without scale or shift: y = (x - mean) / sqrt(var + eps),
// D <= layer_norm_max_d(); x and y [T][D] of the same type.
size_t layer_norm_max_d();
cudaError_t launch_layer_norm(const void* x, int64_t T, int D, float eps, int is_bf16, void* y, cudaStream_t s);
// dx = dout + the layer norm's gradient for g = sum of the n partials G [n][T][D]
// (fp32, summed in order); x and dout [T][D] of the path's type, dx fp32.
cudaError_t launch_layer_norm_bwd(const float* G, int n, const void* x, const void* dout, int64_t T, int D, float eps,
                                  int is_bf16, float* dx, cudaStream_t s);
// out += res, fp32.
cudaError_t launch_add_residual_f32(float* out, const float* res, int64_t count, cudaStream_t s);

// Per-shard descriptor kept in device memory by the shards handle.
struct ShardDesc {
  void* A;   // A_i  [D, Fs]
  void* B;   // B_i  [Fs, D]
  void* At;  // A_i^T [Fs, D] (bf16 only, else null)
  void* Bt;  // B_i^T [D, Fs] (bf16 only, else null)
  int64_t f0;  // first column of A (row of B) owned by the shard
};
// Copies every shard's slices A_i, B_i out of A [D, F] and B [F, D]; the
// destinations come from the device descriptor table.
cudaError_t launch_shard_copy(const void* A, const void* B, const ShardDesc* d_table, int64_t D, int64_t F,
                              int64_t Fs, int elem_bytes, cudaStream_t s);

// out[c, r] = in[r, c] for 2-byte elements; in has row pitch ldi, out ldo.
cudaError_t launch_transpose_u16(const void* in, int64_t rows, int64_t cols, int64_t ldi, void* out, int64_t ldo,
                                 cudaStream_t s);

// fp32 path: H <- GeLU(P) and, in place, dH <- dH * GeLU'(P); count elements.
cudaError_t launch_bwd_act_f32(const float* P, float* H, float* dH, int64_t count, cudaStream_t s);

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t s);
// Debug build only: one block writes element `index` of a 32-element shared
// array behind a device-side check (kChkSelftest).
cudaError_t launch_bounds_selftest(int index, cudaStream_t s);

// Attention of head-split tensor parallelism (attention.cu), per rank i:
// O_i = softmax(Q K^T / sqrt(d_h)) V for each of its local heads and each
// sequence, Q, K, V from the rank's QKV projection. Tensor-core form: bf16,
// d_h = 64, seq % 8 == 0 (the streaming kernel; TPMLP_ATTN_KERNEL=0 selects the
// exact one up to 512 tokens); V read from its transpose.
struct AttnLaunch {
  const CUtensorMap* map_qkv[kMaxGroups];  // QKV_i [T, 3 Dn] bf16, 64 x 128 boxes (make_operand_map, 128 rows)
  const CUtensorMap* map_vt[kMaxGroups];   // V_i^T [Dn, T] bf16, 64 x 64 boxes (make_operand_map, 64 rows)
  void* out[kMaxGroups];                   // O_i [T, Dn] bf16
  int n, batch, seq, Dn, local_heads;
  uint64_t wait_ns;
  int* status;
};
cudaError_t launch_attention_tc(const AttnLaunch& a, cudaStream_t s);
// fp32 form on the CUDA cores: qkv [n][T][3 Dn], out [n][T][Dn]; d_h <= 128, seq <= 8192.
cudaError_t launch_attention_f32(const float* qkv, int64_t T, int n, int Dn, int dh, int local_heads, int batch,
                                 int seq, float* out, cudaStream_t s);

// Device address of the status word that bounded waits write on this device.
int* device_status_word();

// Reads and clears the device status word.
cudaError_t read_and_clear_status(int* value, cudaStream_t s);

int num_sms();

// Programmatic dependent launch (TPMLP_PDL=0 turns it off): the kernels that
// start with pdl_wait() are launched with this, so their set-up overlaps the
// tail of the previous kernel in the stream.
bool pdl_enabled();
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Records the calling thread's error message (what tpmlp_last_error returns)
// and returns `code`.
int set_error(int code, const char* fmt, ...);

}  // namespace tpmlp
