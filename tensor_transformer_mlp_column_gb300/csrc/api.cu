// api.cu — the library's C ABI (include/tpmlp.h): argument checks, the shards
// handle with its descriptor table and tensor maps, workspace planning, and
// the sequence of kernel launches for each call. Nothing here computes on the
// host: every step of the MLP runs in the kernels of gemm_tc.cu, simt.cu and
// elementwise.cu.
#include "tpmlp.h"

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "internal.h"
#include "trace.h"

using namespace tpmlp;

struct tpmlp_shards {
  int device = 0;
  int64_t D = 0, F = 0, Fs = 0;
  int n = 0;
  tpmlp_dtype dt = TPMLP_F32;
  void* mem = nullptr;
  ShardDesc* d_table = nullptr;
  std::vector<ShardDesc> desc;  // host copy of the descriptor table
  // bf16 only: TMA maps of the shard-owned operands, all used as the "N x K"
  // operand of a tensor-core product.
  std::vector<CUtensorMap> map_At;  // A_i^T [Fs, D]: X A_i        (N = Fs, K = D)
  std::vector<CUtensorMap> map_Bt;  // B_i^T [D, Fs]: H_i B_i      (N = D,  K = Fs)
  std::vector<CUtensorMap> map_Bt64;  // the same in 64-row boxes (narrow tiles of a small shard-ordered sum)
  std::vector<CUtensorMap> map_B;   // B_i   [Fs, D]: dY B_i^T     (N = Fs, K = D)
  std::vector<CUtensorMap> map_A;   // A_i   [D, Fs]: dP_i A_i^T   (N = D,  K = Fs)
};

namespace {

thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

#define TRY_CUDA(expr)                                                                        \
  do {                                                                                        \
    cudaError_t e_ = (expr);                                                                  \
    if (e_ != cudaSuccess) return fail(TPMLP_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

// TRY_CUDA of a launch that TPMLP_TRACE=1 times as the step `phase` (trace.cu).
#define TRACED(phase, stream, expr)     \
  do {                                  \
    TraceScope trace_scope_(phase, stream); \
    TRY_CUDA(expr);                     \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
size_t esize(tpmlp_dtype dt) { return dt == TPMLP_BF16 ? 2 : 4; }

// Read once per process (thread-safe static initialisation).
uint64_t wait_limit_ns() {
  static const uint64_t v = [] {
    const char* s = getenv("TPMLP_WAIT_LIMIT_MS");
    long ms = s ? atol(s) : 0;
    if (ms <= 0 || ms > 600000) ms = 4000;
    return static_cast<uint64_t>(ms) * 1000000ull;
  }();
  return v;
}

// The kernels are built for sm_103a only.
int check_device(int* dev_out) {
  int dev = -1;
  TRY_CUDA(cudaGetDevice(&dev));
  int major = 0, minor = 0;
  TRY_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
  TRY_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
  if (major != 10 || minor != 3)
    return fail(TPMLP_ERR_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a (GB300)", dev, major,
                minor);
  if (dev_out) *dev_out = dev;
  return TPMLP_OK;
}

int check_handle_device(const tpmlp_shards* sh) {
  int dev = -1;
  int rc = check_device(&dev);
  if (rc) return rc;
  if (dev != sh->device)
    return fail(TPMLP_ERR_DEVICE, "shards live on device %d but device %d is current", sh->device, dev);
  return TPMLP_OK;
}

// Workspace plan: byte offsets of every scratch buffer, 256-byte aligned.
struct WsPlan {
  size_t H = 0, Yp = 0, P = 0, dH = 0, dP = 0, dXp = 0, bands = 0;
  size_t total = 0;
};

// Whether the bf16 forward runs its two products in one persistent launch
// (gemm_fwd.cu): when both have enough 256 x 256 tiles for CTA pairs (the
// launcher's own rule), together no more than 32 rounds of them over the
// pairs, and all shards' weights (A_i^T and B_i^T, 4 D F bytes) within
// 64 MiB: the one launch walks its tiles band by band (256 token rows), so
// every band streams the whole of the weights, which must stay in L2. There
// one product's partly filled last round and the other's first share the GPU
// and no launch separates them. TPMLP_FWD_PERSIST=0 (read once per process)
// keeps two launches for comparisons.
bool use_persistent_forward(int64_t T, const tpmlp_shards* sh, tpmlp_mode mode) {
  static const bool on = [] {
    const char* e = getenv("TPMLP_FWD_PERSIST");
    return !(e && *e && atoi(e) == 0);
  }();
  if (!on || sh->dt != TPMLP_BF16 || !tc_pairs_enabled()) return false;
  const int64_t mb = (T + 255) / 256;
  const int64_t t1 = mb * ((sh->Fs + 255) / 256) * sh->n;
  const int chain = mode == TPMLP_FUSED ? 1 : 0;
  const int w2 = fwd_second_width(T, sh->D, chain);
  const int64_t t2 = mb * ((sh->D + w2 - 1) / w2) * (chain ? 1 : sh->n);
  const int64_t sms = num_sms();
  const int pairs = fwd_persistent_clusters();
  const int64_t weight_bytes = 4 * sh->D * static_cast<int64_t>(sh->Fs) * sh->n;
  return pairs > 0 && t1 >= sms / 4 && t2 >= sms / 4 && t1 + t2 <= 32 * static_cast<int64_t>(pairs) &&
         weight_bytes <= (int64_t(64) << 20);
}

// Whether the bf16 recomputing backward runs its first step in the dual
// kernel (gemm_dual.cu: P_i and dH_i in tensor memory, P never written): for
// products with enough 256 x 256 tiles to keep CTA pairs busy, as the other
// tensor-core products decide (TPMLP_BWD_DUAL=0 computes P_i into the
// workspace with one product and applies the activation in the epilogue of
// the dH_i product instead, for comparisons; read once per process).
bool use_dual_backward(int64_t T, const tpmlp_shards* sh) {
  static const bool on = [] {
    const char* e = getenv("TPMLP_BWD_DUAL");
    return !(e && *e && atoi(e) == 0);
  }();
  if (!on || sh->dt != TPMLP_BF16 || !tc_pairs_enabled()) return false;
  const int64_t tiles = ((T + 255) / 256) * ((sh->Fs + 255) / 256) * sh->n;
  return tiles >= num_sms() / 4;
}

WsPlan plan_workspace(int64_t T, const tpmlp_shards* sh, tpmlp_mode mode, int backward) {
  WsPlan w;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, 256);
    return at;
  };
  const size_t n = sh->n, D = sh->D, Fs = sh->Fs, t = T, es = esize(sh->dt);
  if (!backward) {
    w.H = take(n * t * Fs * es);
    if (mode == TPMLP_FAITHFUL) w.Yp = take(n * t * D * 4);
    if (use_persistent_forward(T, sh, mode)) w.bands = take(((t + 255) / 256) * sizeof(int));
  } else {
    // backward == 2: the caller's saved P; the dual kernel keeps P in tensor memory.
    if (backward == 1 && !use_dual_backward(T, sh)) w.P = take(n * t * Fs * 4);
    if (sh->dt == TPMLP_F32) {  // bf16 applies the activation in a product's epilogue instead
      w.H = take(n * t * Fs * 4);
      w.dH = take(n * t * Fs * 4);
    } else {
      w.H = take(n * t * Fs * 2);
      w.dP = take(n * t * Fs * 2);
    }
    if (mode == TPMLP_FAITHFUL) w.dXp = take(n * t * D * 4);
  }
  w.total = off;
  return w;
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

int map_or_fail(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t pitch, int box_rows,
                const char* what) {
  if (!make_operand_map(m, base, rows, cols, pitch, box_rows))
    return fail(TPMLP_ERR_CUDA, "cuTensorMapEncodeTiled rejected the map of %s [%lld x %lld]", what,
                static_cast<long long>(rows), static_cast<long long>(cols));
  return TPMLP_OK;
}

// Map of a row-major bf16 [rows][cols] tensor read as an MN-major operand of
// a product that contracts over its rows: a 3-D map (one TMA box per 128
// columns) where cols is a multiple of 64, else a 2-D one in 64 x 64 boxes.
// Adds the matching TcMajor bits (kMnA/kMnA3d, or kMnB/kMnB3d with is_b) to *major.
int mn_map_or_fail(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t pitch, bool is_b,
                   int* major, const char* what) {
  *major |= is_b ? kMnB : kMnA;
  if (cols % 64 == 0 && make_operand_map_mn3d(m, base, rows, cols, pitch)) {
    *major |= is_b ? kMnB3d : kMnA3d;
    return TPMLP_OK;
  }
  return map_or_fail(m, base, rows, cols, pitch, 64, what);
}

int out_map(CUtensorMap* m, void* base, int64_t rows, int64_t cols, int64_t pitch, const char* what) {
  if (!make_output_map_f32(m, base, rows, cols, pitch))
    return fail(TPMLP_ERR_CUDA, "cuTensorMapEncodeTiled rejected the output map of %s [%lld x %lld]", what,
                static_cast<long long>(rows), static_cast<long long>(cols));
  return TPMLP_OK;
}

// ----------------------------------------------------------- step launchers

// H_i = GeLU(X A_i) for every shard, and with P_out also P_i = X A_i (fp32,
// [n][T][Fs]). `inject` and `wait_ns` are the test hooks of
// tpmlp_selftest_gemm_withheld_fill (0 = off / the default limit).
int run_hidden(const void* X, int64_t T, const tpmlp_shards* sh, void* H, cudaStream_t s, int inject = 0,
               uint64_t wait_ns = 0, void* P_out = nullptr) {
  const int64_t D = sh->D, Fs = sh->Fs;
  if (sh->dt == TPMLP_BF16) {
    CUtensorMap mx;
    std::vector<CUtensorMap> mo(sh->n);
    int rc = map_or_fail(&mx, X, T, D, D, tc_box_rows_a(), "X");
    if (rc) return rc;
    TcGemm g{};
    g.groups = sh->n;
    for (int i = 0; i < sh->n; ++i) {
      g.map_a[i] = &mx;
      g.map_b[i] = &sh->map_At[i];
      g.out[i] = at<uint16_t>(H, 0) + static_cast<size_t>(i) * T * Fs;
      if (P_out) {
        g.out2[i] = static_cast<float*>(P_out) + static_cast<size_t>(i) * T * Fs;
      } else {
        // H_i leaves the pair kernel through TMA stores.
        if (!make_output_map_bf16(&mo[i], g.out[i], T, Fs, Fs))
          return fail(TPMLP_ERR_CUDA, "cuTensorMapEncodeTiled rejected the output map of H_%d [%lld x %lld]", i,
                      static_cast<long long>(T), static_cast<long long>(Fs));
        g.map_out[i] = &mo[i];
      }
    }
    g.ldo = Fs;
    g.M = static_cast<int>(T);
    g.N = static_cast<int>(Fs);
    g.K = static_cast<int>(D);
    g.epi = P_out ? kEpiGeluSaveP : kEpiGeluBf16;
    g.shared = kSharedA;  // X feeds every shard
    g.group_m = 16;       // bands of 16 M blocks: fewest DRAM re-reads of the shards' A_i^T measured
    g.stream_out = 1;
    g.inject = inject;
    TRACED(P_out ? "gemm1_gelu_save_p" : "gemm1_gelu", s, launch_tc_gemm(g, wait_ns ? wait_ns : wait_limit_ns(), s));
    return TPMLP_OK;
  }
  for (int i = 0; i < sh->n; ++i) {
    float* Ci = static_cast<float*>(P_out ? P_out : H) + static_cast<size_t>(i) * T * Fs;
    SimtGemm g{static_cast<const float*>(X), D, 1, static_cast<const float*>(sh->desc[i].A), Fs, 1, Ci, Fs,
               static_cast<int>(T), static_cast<int>(Fs), static_cast<int>(D), P_out ? kSimtStore : kSimtGelu};
    TRY_CUDA(launch_simt_gemm(g, s));
  }
  if (P_out) TRY_CUDA(launch_gelu(P_out, H, static_cast<int64_t>(sh->n) * T * Fs, 0, s));  // H = GeLU(P)
  return TPMLP_OK;
}

// Y_i = H_i B_i into Yp (chain = 0), or Y = sum_i H_i B_i into Y (chain = 1);
// with chain = 1 and a residual R [T][D] of the path's type, Y = R + that sum.
// With slices (chain = 1 only), the output rows are cut into n rank slices of
// T/n rows and slice j goes to slices->p[j] instead of `out`.
int run_second(const void* H, int64_t T, const tpmlp_shards* sh, void* out, int chain, cudaStream_t s,
               const void* resid = nullptr, const OutSlices* slices = nullptr) {
  const int64_t D = sh->D, Fs = sh->Fs;
  if (sh->dt == TPMLP_BF16) {
    std::vector<CUtensorMap> mh(sh->n), mo(sh->n);
    TcGemm g{};
    g.groups = sh->n;
    for (int i = 0; i < sh->n; ++i) {
      int rc = map_or_fail(&mh[i], at<uint16_t>(const_cast<void*>(H), 0) + static_cast<size_t>(i) * T * Fs, T, Fs,
                           Fs, tc_box_rows_a(), "H_i");
      if (rc) return rc;
      g.map_a[i] = &mh[i];
      g.map_b[i] = &sh->map_Bt[i];
      if (chain) g.map_b_narrow[i] = &sh->map_Bt64[i];
      if (slices) {  // rank slices: one output (and output map) per slice of T/n rows
        g.out[i] = slices->p[i];
        if ((rc = out_map(&mo[i], g.out[i], T / sh->n, D, D, "Y slice"))) return rc;
        g.map_out[i] = &mo[i];
        continue;
      }
      g.out[i] = chain ? out : static_cast<void*>(static_cast<float*>(out) + static_cast<size_t>(i) * T * D);
      if ((rc = out_map(&mo[i], g.out[i], T, D, D, "Y_i"))) return rc;
      g.map_out[i] = &mo[i];
    }
    if (slices) g.slice_rows = T / sh->n;
    g.ldo = D;
    g.M = static_cast<int>(T);
    g.N = static_cast<int>(D);
    g.K = static_cast<int>(Fs);
    g.chain = chain;
    g.epi = kEpiF32;
    g.group_m = 8;
    g.stream_out = 1;
    g.resid = chain ? resid : nullptr;
    TRACED(chain ? "gemm2_fused_sum" : "gemm2_partials", s, launch_tc_gemm(g, wait_limit_ns(), s));
    return TPMLP_OK;
  }
  // fp32: one product per shard (and, with rank slices, per slice of T/n rows).
  const int nsl = slices ? sh->n : 1;
  const int64_t rows = T / nsl;
  for (int j = 0; j < nsl; ++j) {
    for (int i = 0; i < sh->n; ++i) {
      float* C = slices ? slices->p[j]
                        : (chain ? static_cast<float*>(out) : static_cast<float*>(out) + static_cast<size_t>(i) * T * D);
      SimtGemm g{static_cast<const float*>(H) + static_cast<size_t>(i) * T * Fs + static_cast<size_t>(j) * rows * Fs,
                 Fs, 1, static_cast<const float*>(sh->desc[i].B), D, 1, C, D, static_cast<int>(rows),
                 static_cast<int>(D), static_cast<int>(Fs), (chain && i > 0) ? kSimtAccumulate : kSimtStore};
      TRY_CUDA(launch_simt_gemm(g, s));
    }
  }
  if (chain && resid)
    TRY_CUDA(launch_add_residual_f32(static_cast<float*>(out), static_cast<const float*>(resid), T * D, s));
  return TPMLP_OK;
}

int check_common(const tpmlp_shards* sh, int64_t T);

// The block's backward tail: the input gradient of the MLP (its shard
// partials, or their sum) goes back through the layer norm of x and picks up
// the residual's dout: dx = dout + LN'(x)^T g.
struct LnTail {
  const void* x;
  const void* dout;
  float eps;
  float* dx;
};

// Workspace of the block calls: LN(x), in FUSED backward the summed MLP input
// gradient, then the MLP call's own workspace.
struct BlockPlan {
  size_t xn = 0, dxn = 0, inner = 0, total = 0;
  WsPlan w;
};

BlockPlan plan_block(int64_t T, const tpmlp_shards* sh, tpmlp_mode mode, int backward) {
  BlockPlan b;
  const size_t td = static_cast<size_t>(T) * sh->D;
  b.xn = 0;
  size_t off = round_up(td * esize(sh->dt), 256);
  if (backward && mode == TPMLP_FUSED) {
    b.dxn = off;
    off = round_up(off + td * 4, 256);
  }
  b.inner = off;
  b.w = plan_workspace(T, sh, mode, backward ? 1 : 0);
  b.total = off + b.w.total;
  return b;
}

// Workspace of the sequence-parallel calls: the all-gathered X (and dY), then
// the MLP call's own workspace.
struct SpPlan {
  size_t x = 0, dy = 0, inner = 0, total = 0;
  WsPlan w;
};

SpPlan plan_sp(int64_t T, const tpmlp_shards* sh, tpmlp_mode mode, int backward) {
  SpPlan p;
  const size_t bytes = static_cast<size_t>(T) * sh->D * esize(sh->dt);
  size_t off = round_up(bytes, 256);
  if (backward) {
    p.dy = off;
    off = round_up(off + bytes, 256);
  }
  p.inner = off;
  p.w = plan_workspace(T, sh, mode, backward ? 1 : 0);
  p.total = off + p.w.total;
  return p;
}

// Checks a host array of n rank-slice pointers (non-NULL, 16-byte aligned).
int check_slices(const void* const* p, int n, const char* what) {
  if (!p) return fail(TPMLP_ERR_ARG, "%s must not be NULL", what);
  for (int j = 0; j < n; ++j) {
    if (!p[j]) return fail(TPMLP_ERR_ARG, "%s[%d] is NULL", what, j);
    if (!aligned16(p[j])) return fail(TPMLP_ERR_ALIGN, "%s[%d] must be 16-byte aligned", what, j);
  }
  return TPMLP_OK;
}

int check_eps(float eps) {
  if (!(eps > 0.f) || !(eps < 1e30f)) return fail(TPMLP_ERR_ARG, "eps = %g must be positive and finite", double(eps));
  return TPMLP_OK;
}

// The bf16 forward's two products in one persistent launch: H_i into H, then
// Y (Yp == NULL: the shard-ordered sum) or the partials Yp. band_extra and
// wait_ns are the test hooks of tpmlp_selftest_forward_band_timeout (0 = off /
// the default limit).
int run_forward_persistent(const void* X, int64_t T, const tpmlp_shards* sh, void* Y, float* Yp, void* H,
                           int* bands, cudaStream_t stream, int band_extra = 0, uint64_t wait_ns = 0) {
  const int64_t D = sh->D, Fs = sh->Fs;
  const int n = sh->n;
  int rc;
  CUtensorMap mx;
  std::vector<CUtensorMap> mh(n), mo(n);
  if ((rc = map_or_fail(&mx, X, T, D, D, tc_box_rows_a(), "X"))) return rc;
  FwdPersistent f{};
  f.map_x = &mx;
  for (int i = 0; i < n; ++i) {
    f.h[i] = at<uint16_t>(H, 0) + static_cast<size_t>(i) * T * Fs;
    if ((rc = map_or_fail(&mh[i], f.h[i], T, Fs, Fs, tc_box_rows_a(), "H_i"))) return rc;
    f.map_at[i] = &sh->map_At[i];
    f.map_h[i] = &mh[i];
    f.map_bt[i] = &sh->map_Bt[i];
    f.map_bt64[i] = &sh->map_Bt64[i];
    void* out = Yp ? static_cast<void*>(Yp + static_cast<size_t>(i) * T * D) : Y;
    if ((i == 0 || Yp) && (rc = out_map(&mo[i], out, T, D, D, Yp ? "Y_i" : "Y"))) return rc;
    f.map_out[i] = &mo[Yp ? i : 0];
  }
  f.M = static_cast<int>(T);
  f.N1 = static_cast<int>(Fs);
  f.N2 = static_cast<int>(D);
  f.K1 = static_cast<int>(D);
  f.groups = n;
  f.chain = Yp ? 0 : 1;
  f.band_done = bands;
  f.band_extra = band_extra;
  TRACED("forward_persistent", stream, launch_fwd_persistent(f, wait_ns ? wait_ns : wait_limit_ns(), stream));
  return TPMLP_OK;
}

// tpmlp_forward, and with P also tpmlp_forward_save.
int forward_impl(const void* X, int64_t T, const tpmlp_shards* sh, void* Y, void* P, tpmlp_mode mode, void* ws,
                 size_t ws_bytes, cudaStream_t stream) {
  int rc = check_common(sh, T);
  if (rc) return rc;
  if (mode != TPMLP_FAITHFUL && mode != TPMLP_FUSED) return fail(TPMLP_ERR_ARG, "unknown mode %d", int(mode));
  if (!X || !Y || !ws) return fail(TPMLP_ERR_ARG, "X, Y and workspace must not be NULL");
  if (!aligned16(X) || !aligned16(Y) || !aligned16(ws))
    return fail(TPMLP_ERR_ALIGN, "X, Y and workspace must be 16-byte aligned");
  const WsPlan w = plan_workspace(T, sh, mode, 0);
  if (ws_bytes < w.total)
    return fail(TPMLP_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, w.total);
  if ((rc = check_handle_device(sh))) return rc;
  void* H = at<char>(ws, w.H);
  float* Yp = mode == TPMLP_FAITHFUL ? at<float>(ws, w.Yp) : nullptr;
  if (!P && use_persistent_forward(T, sh, mode)) {
    // Both products in one launch; the second product's tiles start on bands
    // of H as they are completed.
    if ((rc = run_forward_persistent(X, T, sh, Y, Yp, H, at<int>(ws, w.bands), stream))) return rc;
    if (!Yp) return TPMLP_OK;
    TRACED("allreduce", stream, launch_allreduce(Yp, sh->n, T * sh->D, static_cast<float*>(Y), stream));
    return TPMLP_OK;
  }
  if ((rc = run_hidden(X, T, sh, H, stream, 0, 0, P))) return rc;
  if (mode == TPMLP_FUSED) return run_second(H, T, sh, Y, 1, stream);
  if ((rc = run_second(H, T, sh, Yp, 0, stream))) return rc;
  TRACED("allreduce", stream, launch_allreduce(Yp, sh->n, T * sh->D, static_cast<float*>(Y), stream));
  return TPMLP_OK;
}

// The last step of the backward: dX = the shard-ordered sum of the partials
// (FAITHFUL; FUSED already accumulated dX), or with a tail the block's dx.
int finish_dx(const float* dXp, int n, int64_t T, const tpmlp_shards* sh, void* dX, const LnTail* tail,
              const OutSlices* slices, cudaStream_t s) {
  if (slices) {  // the rank slices were written by the product (fused) or come from the partials
    if (dXp) TRACED("bwd_dx_reduce_scatter", s, launch_reduce_scatter(dXp, n, T * sh->D, *slices, n, s));
    return TPMLP_OK;
  }
  if (tail) {
    const float* G = dXp ? dXp : static_cast<const float*>(dX);
    TRACED("bwd_layer_norm_tail", s, launch_layer_norm_bwd(G, dXp ? n : 1, tail->x, tail->dout, T, static_cast<int>(sh->D), tail->eps,
                                   sh->dt == TPMLP_BF16, tail->dx, s));
    return TPMLP_OK;
  }
  if (dXp) TRACED("bwd_dx_allreduce", s, launch_allreduce(dXp, n, T * sh->D, static_cast<float*>(dX), s));
  return TPMLP_OK;
}

int check_common(const tpmlp_shards* sh, int64_t T) {
  if (!sh) return fail(TPMLP_ERR_ARG, "shards handle is NULL");
  if (T < 1) return fail(TPMLP_ERR_ARG, "T = %lld must be >= 1", static_cast<long long>(T));
  if (T > (int64_t(1) << 30)) return fail(TPMLP_ERR_ARG, "T = %lld is too large", static_cast<long long>(T));
  return TPMLP_OK;
}

}  // namespace

int tpmlp::set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

extern "C" {

int tpmlp_version(void) { return (1 << 16) | 0; }

const char* tpmlp_last_error(void) { return g_msg; }

int tpmlp_check_status(tpmlp_stream_t stream) {
  int v = 0;
  TRY_CUDA(read_and_clear_status(&v, stream));
  if (v == kSiteSmemAlign)
    return fail(TPMLP_ERR_CUDA, "a kernel found its dynamic shared memory misaligned and did no work");
  if (v >= kSiteBoundsBase) {
    static const char* const kNames[kChkCount] = {
        "?", "GEMM tile outside the tile grid", "TMA coordinate not 16-byte aligned", "epilogue store outside the output",
        "reduce index outside its slice", "attention tile outside the launch", "self-test index outside its array"};
    const int c = v - kSiteBoundsBase;
    return fail(TPMLP_ERR_BOUNDS, "a device-side check failed: %s (check %d)", c > 0 && c < kChkCount ? kNames[c] : "?",
                c);
  }
  if (v) return fail(TPMLP_ERR_TIMEOUT, "a device-side wait ran out of time (site %d)", v);
  return TPMLP_OK;
}

int tpmlp_build_flags(void) { return kDebugBuild ? 1 : 0; }

int tpmlp_selftest_bounds(int index, tpmlp_stream_t stream) {
  if (!kDebugBuild) return fail(TPMLP_ERR_UNSUPPORTED, "the device-side checks exist in the debug build only");
  int rc = check_device(nullptr);
  if (rc) return rc;
  TRY_CUDA(launch_bounds_selftest(index, stream));
  return TPMLP_OK;
}

int tpmlp_gelu(const void* x, void* y, int64_t n, tpmlp_dtype dt, tpmlp_stream_t stream) {
  if (n < 0) return fail(TPMLP_ERR_ARG, "n = %lld must be >= 0", static_cast<long long>(n));
  if (dt != TPMLP_F32 && dt != TPMLP_BF16) return fail(TPMLP_ERR_ARG, "unknown dtype %d", int(dt));
  if (n == 0) return TPMLP_OK;
  if (!x || !y) return fail(TPMLP_ERR_ARG, "x and y must not be NULL");
  if (!aligned16(x) || !aligned16(y)) return fail(TPMLP_ERR_ALIGN, "x and y must be 16-byte aligned");
  int rc = check_device(nullptr);
  if (rc) return rc;
  TRACED("gelu", stream, launch_gelu(x, y, n, dt == TPMLP_BF16, stream));
  return TPMLP_OK;
}

int tpmlp_shard(const void* A, const void* B, int64_t D, int64_t F, int n, tpmlp_dtype dt, tpmlp_stream_t stream,
                tpmlp_shards** out) {
  if (!out) return fail(TPMLP_ERR_ARG, "out must not be NULL");
  *out = nullptr;
  if (!A || !B) return fail(TPMLP_ERR_ARG, "A and B must not be NULL");
  if (D < 1 || F < 1) return fail(TPMLP_ERR_ARG, "D and F must be >= 1");
  if (n < 1) return fail(TPMLP_ERR_ARG, "n = %d must be >= 1", n);
  if (dt != TPMLP_F32 && dt != TPMLP_BF16) return fail(TPMLP_ERR_ARG, "unknown dtype %d", int(dt));
  if (F % n != 0)
    return fail(TPMLP_ERR_DIVISIBILITY, "F = %lld is not divisible by n = %d", static_cast<long long>(F), n);
  const int64_t Fs = F / n;
  if (dt == TPMLP_BF16) {
    if (n > TPMLP_MAX_SHARDS)
      return fail(TPMLP_ERR_UNSUPPORTED, "bf16 supports at most %d shards, got %d", TPMLP_MAX_SHARDS, n);
    if (D % 8 != 0 || Fs % 8 != 0)
      return fail(TPMLP_ERR_SHAPE, "bf16 needs D and F/n to be multiples of 8 (D = %lld, F/n = %lld)",
                  static_cast<long long>(D), static_cast<long long>(Fs));
    if (D > (int64_t(1) << 30) || Fs > (int64_t(1) << 30)) return fail(TPMLP_ERR_SHAPE, "D or F/n too large");
  }
  if (!aligned16(A) || !aligned16(B)) return fail(TPMLP_ERR_ALIGN, "A and B must be 16-byte aligned");
  int dev = -1;
  int rc = check_device(&dev);
  if (rc) return rc;

  tpmlp_shards* sh = new tpmlp_shards();
  sh->device = dev;
  sh->D = D;
  sh->F = F;
  sh->Fs = Fs;
  sh->n = n;
  sh->dt = dt;
  const size_t es = esize(dt), blk = round_up(static_cast<size_t>(D) * Fs * es, 256);
  const int layouts = dt == TPMLP_BF16 ? 4 : 2;
  cudaError_t e = cudaMalloc(&sh->mem, blk * layouts * n);
  if (e == cudaSuccess) e = cudaMalloc(&sh->d_table, sizeof(ShardDesc) * n);
  if (e != cudaSuccess) {
    tpmlp_shards_free(sh);
    return fail(TPMLP_ERR_CUDA, "cudaMalloc of the shards failed: %s", cudaGetErrorString(e));
  }
  sh->desc.resize(n);
  for (int i = 0; i < n; ++i) {
    char* base = static_cast<char*>(sh->mem) + blk * layouts * i;  // shard i's own block
    sh->desc[i].A = base;
    sh->desc[i].B = base + blk;
    sh->desc[i].At = layouts == 4 ? base + 2 * blk : nullptr;
    sh->desc[i].Bt = layouts == 4 ? base + 3 * blk : nullptr;
    sh->desc[i].f0 = i * Fs;
  }
  e = cudaMemcpyAsync(sh->d_table, sh->desc.data(), sizeof(ShardDesc) * n, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = launch_shard_copy(A, B, sh->d_table, D, F, Fs, static_cast<int>(es), stream);
  if (dt == TPMLP_BF16) {
    for (int i = 0; i < n && e == cudaSuccess; ++i) {
      e = launch_transpose_u16(sh->desc[i].A, D, Fs, Fs, sh->desc[i].At, D, stream);  // A_i^T [Fs, D]
      if (e == cudaSuccess) e = launch_transpose_u16(sh->desc[i].B, Fs, D, D, sh->desc[i].Bt, Fs, stream);  // B_i^T
    }
  }
  if (e != cudaSuccess) {
    cudaStreamSynchronize(stream);
    tpmlp_shards_free(sh);
    return fail(TPMLP_ERR_CUDA, "shard copy failed: %s", cudaGetErrorString(e));
  }
  if (dt == TPMLP_BF16) {
    sh->map_At.resize(n);
    sh->map_Bt.resize(n);
    sh->map_Bt64.resize(n);
    sh->map_B.resize(n);
    sh->map_A.resize(n);
    for (int i = 0; i < n; ++i) {
      const ShardDesc& d = sh->desc[i];
      rc = map_or_fail(&sh->map_At[i], d.At, Fs, D, D, tc_box_rows_b(static_cast<int>(Fs)), "A_i^T");
      if (!rc) rc = map_or_fail(&sh->map_Bt[i], d.Bt, D, Fs, Fs, tc_box_rows_b(static_cast<int>(D)), "B_i^T");
      if (!rc) rc = map_or_fail(&sh->map_Bt64[i], d.Bt, D, Fs, Fs, 64, "B_i^T");
      if (!rc) rc = map_or_fail(&sh->map_B[i], d.B, Fs, D, D, tc_box_rows_b(static_cast<int>(Fs)), "B_i");
      if (!rc) rc = map_or_fail(&sh->map_A[i], d.A, D, Fs, Fs, tc_box_rows_b(static_cast<int>(D)), "A_i");
      if (rc) {
        cudaStreamSynchronize(stream);
        tpmlp_shards_free(sh);
        return rc;
      }
    }
  }
  *out = sh;
  return TPMLP_OK;
}

int tpmlp_shard_info(const tpmlp_shards* sh, int64_t* D, int64_t* F, int* n, tpmlp_dtype* dt) {
  if (!sh) return fail(TPMLP_ERR_ARG, "shards handle is NULL");
  if (D) *D = sh->D;
  if (F) *F = sh->F;
  if (n) *n = sh->n;
  if (dt) *dt = sh->dt;
  return TPMLP_OK;
}

int tpmlp_shard_get(const tpmlp_shards* sh, int i, const void** A_i, const void** B_i) {
  if (!sh) return fail(TPMLP_ERR_ARG, "shards handle is NULL");
  if (i < 0 || i >= sh->n) return fail(TPMLP_ERR_ARG, "shard index %d out of range [0, %d)", i, sh->n);
  if (A_i) *A_i = sh->desc[i].A;
  if (B_i) *B_i = sh->desc[i].B;
  return TPMLP_OK;
}

int tpmlp_shard_get_transposed(const tpmlp_shards* sh, int i, const void** At_i, const void** Bt_i) {
  if (!sh) return fail(TPMLP_ERR_ARG, "shards handle is NULL");
  if (i < 0 || i >= sh->n) return fail(TPMLP_ERR_ARG, "shard index %d out of range [0, %d)", i, sh->n);
  if (sh->dt != TPMLP_BF16) return fail(TPMLP_ERR_UNSUPPORTED, "fp32 shards keep no transposed copies");
  if (At_i) *At_i = sh->desc[i].At;
  if (Bt_i) *Bt_i = sh->desc[i].Bt;
  return TPMLP_OK;
}

void tpmlp_shards_free(tpmlp_shards* sh) {
  if (!sh) return;
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != sh->device) cudaSetDevice(sh->device);
  cudaDeviceSynchronize();
  if (sh->mem) cudaFree(sh->mem);
  if (sh->d_table) cudaFree(sh->d_table);
  if (prev >= 0 && prev != sh->device) cudaSetDevice(prev);
  delete sh;
}

size_t tpmlp_workspace_bytes(int64_t T, const tpmlp_shards* sh, tpmlp_mode mode, int backward) {
  if (!sh || T < 1 || (mode != TPMLP_FAITHFUL && mode != TPMLP_FUSED) || backward < 0 || backward > 2) return 0;
  return plan_workspace(T, sh, mode, backward).total;
}

int tpmlp_hidden(const void* X, int64_t T, const tpmlp_shards* sh, void* H, tpmlp_stream_t stream) {
  int rc = check_common(sh, T);
  if (rc) return rc;
  if (!X || !H) return fail(TPMLP_ERR_ARG, "X and H must not be NULL");
  if (!aligned16(X) || !aligned16(H)) return fail(TPMLP_ERR_ALIGN, "X and H must be 16-byte aligned");
  if ((rc = check_handle_device(sh))) return rc;
  return run_hidden(X, T, sh, H, stream);
}

int tpmlp_partials(const void* H, int64_t T, const tpmlp_shards* sh, void* Yp, tpmlp_stream_t stream) {
  int rc = check_common(sh, T);
  if (rc) return rc;
  if (!H || !Yp) return fail(TPMLP_ERR_ARG, "H and Yp must not be NULL");
  if (!aligned16(H) || !aligned16(Yp)) return fail(TPMLP_ERR_ALIGN, "H and Yp must be 16-byte aligned");
  if ((rc = check_handle_device(sh))) return rc;
  return run_second(H, T, sh, Yp, 0, stream);
}

int tpmlp_allreduce(const void* Yp, int n, int64_t count, void* Y, tpmlp_stream_t stream) {
  if (n < 1) return fail(TPMLP_ERR_ARG, "n = %d must be >= 1", n);
  if (count < 0) return fail(TPMLP_ERR_ARG, "count must be >= 0");
  if (count == 0) return TPMLP_OK;
  if (!Yp || !Y) return fail(TPMLP_ERR_ARG, "Yp and Y must not be NULL");
  if (!aligned16(Yp) || !aligned16(Y)) return fail(TPMLP_ERR_ALIGN, "Yp and Y must be 16-byte aligned");
  int rc = check_device(nullptr);
  if (rc) return rc;
  TRACED("allreduce", stream, launch_allreduce(static_cast<const float*>(Yp), n, count, static_cast<float*>(Y), stream));
  return TPMLP_OK;
}

int tpmlp_fused_sum(const void* H, int64_t T, const tpmlp_shards* sh, void* Y, tpmlp_stream_t stream) {
  int rc = check_common(sh, T);
  if (rc) return rc;
  if (!H || !Y) return fail(TPMLP_ERR_ARG, "H and Y must not be NULL");
  if (!aligned16(H) || !aligned16(Y)) return fail(TPMLP_ERR_ALIGN, "H and Y must be 16-byte aligned");
  if ((rc = check_handle_device(sh))) return rc;
  return run_second(H, T, sh, Y, 1, stream);
}

int tpmlp_forward(const void* X, int64_t T, const tpmlp_shards* sh, void* Y, tpmlp_mode mode, void* ws,
                  size_t ws_bytes, tpmlp_stream_t stream) {
  return forward_impl(X, T, sh, Y, nullptr, mode, ws, ws_bytes, stream);
}

int tpmlp_forward_save(const void* X, int64_t T, const tpmlp_shards* sh, void* Y, void* P, tpmlp_mode mode, void* ws,
                       size_t ws_bytes, tpmlp_stream_t stream) {
  if (!P) return fail(TPMLP_ERR_ARG, "P must not be NULL");
  if (!aligned16(P)) return fail(TPMLP_ERR_ALIGN, "P must be 16-byte aligned");
  return forward_impl(X, T, sh, Y, P, mode, ws, ws_bytes, stream);
}

static int backward_impl(const void* X, const void* dY, const void* P_saved, int64_t T, const tpmlp_shards* sh,
                         void* dX, void* const* dA, void* const* dB, tpmlp_mode mode, void* ws, size_t ws_bytes,
                         cudaStream_t stream, const LnTail* tail, const OutSlices* dx_slices = nullptr);

int tpmlp_backward(const void* X, const void* dY, int64_t T, const tpmlp_shards* sh, void* dX, void* const* dA,
                   void* const* dB, tpmlp_mode mode, void* ws, size_t ws_bytes, tpmlp_stream_t stream) {
  return backward_impl(X, dY, nullptr, T, sh, dX, dA, dB, mode, ws, ws_bytes, stream, nullptr);
}

int tpmlp_backward_saved(const void* X, const void* dY, const void* P, int64_t T, const tpmlp_shards* sh, void* dX,
                         void* const* dA, void* const* dB, tpmlp_mode mode, void* ws, size_t ws_bytes,
                         tpmlp_stream_t stream) {
  if (!P) return fail(TPMLP_ERR_ARG, "P must not be NULL");
  if (!aligned16(P)) return fail(TPMLP_ERR_ALIGN, "P must be 16-byte aligned");
  return backward_impl(X, dY, P, T, sh, dX, dA, dB, mode, ws, ws_bytes, stream, nullptr);
}

// tpmlp_backward (P_saved == NULL: P_i = X A_i is recomputed into the
// workspace) and tpmlp_backward_saved (P_saved is the forward's P, only read).
// With a tail (tpmlp_block_backward), X is the normalised block input, and
// the input gradient is finished by the tail kernel instead of the reduce:
// from the partials in FAITHFUL mode, from dX (then a scratch buffer) in
// FUSED mode.
// The recomputing backward's first step in the dual kernel: H_i = GeLU(X A_i)
// and dP_i = dY B_i^T * GeLU'(X A_i) into H and dP (bf16 [n][T][Fs]). inject
// and wait_ns are the test hooks of tpmlp_selftest_backward_withheld_fill
// (0 = off / the default limit).
static int run_dual(const CUtensorMap* mX, const CUtensorMap* mdY, int64_t T, const tpmlp_shards* sh, uint16_t* H,
                    uint16_t* dP, cudaStream_t s, int inject = 0, uint64_t wait_ns = 0) {
  const int n = sh->n;
  const int64_t Fs = sh->Fs;
  DualBwd d{};
  d.map_x = mX;
  d.map_dy = mdY;
  for (int i = 0; i < n; ++i) {
    d.map_at[i] = &sh->map_At[i];
    d.map_b[i] = &sh->map_B[i];
    d.h[i] = H + static_cast<size_t>(i) * T * Fs;
    d.dp[i] = dP + static_cast<size_t>(i) * T * Fs;
  }
  d.ldo = Fs;
  d.M = static_cast<int>(T);
  d.N = static_cast<int>(Fs);
  d.K = static_cast<int>(sh->D);
  d.groups = n;
  d.group_m = 16;  // X and dY feed every shard
  d.load_hint = 1 | (1 << 2);
  d.inject = inject;
  TRACED("bwd_dual_P_dH", s, launch_dual_bwd(d, wait_ns ? wait_ns : wait_limit_ns(), s));
  return TPMLP_OK;
}

static int backward_impl(const void* X, const void* dY, const void* P_saved, int64_t T, const tpmlp_shards* sh,
                         void* dX, void* const* dA, void* const* dB, tpmlp_mode mode, void* ws, size_t ws_bytes,
                         cudaStream_t stream, const LnTail* tail, const OutSlices* dx_slices) {
  int rc = check_common(sh, T);
  if (rc) return rc;
  if (mode != TPMLP_FAITHFUL && mode != TPMLP_FUSED) return fail(TPMLP_ERR_ARG, "unknown mode %d", int(mode));
  if (!X || !dY || !dX || !dA || !dB || !ws) return fail(TPMLP_ERR_ARG, "a required pointer is NULL");
  if (!aligned16(X) || !aligned16(dY) || !aligned16(dX) || !aligned16(ws))
    return fail(TPMLP_ERR_ALIGN, "X, dY, dX and workspace must be 16-byte aligned");
  for (int i = 0; i < sh->n; ++i) {
    if (!dA[i] || !dB[i]) return fail(TPMLP_ERR_ARG, "dA[%d] or dB[%d] is NULL", i, i);
    if (!aligned16(dA[i]) || !aligned16(dB[i])) return fail(TPMLP_ERR_ALIGN, "dA[%d], dB[%d] must be 16-byte aligned", i, i);
  }
  const WsPlan w = plan_workspace(T, sh, mode, P_saved ? 2 : 1);
  if (ws_bytes < w.total)
    return fail(TPMLP_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, w.total);
  if ((rc = check_handle_device(sh))) return rc;
  const int n = sh->n;
  const int64_t D = sh->D, Fs = sh->Fs;
  // P_i = X A_i: the caller's (only read) or recomputed here into the workspace.
  float* P = P_saved ? const_cast<float*>(static_cast<const float*>(P_saved)) : at<float>(ws, w.P);
  float* dH = at<float>(ws, w.dH);
  float* dXp = mode == TPMLP_FAITHFUL ? at<float>(ws, w.dXp) : nullptr;
  cudaStream_t s = stream;

  if (sh->dt == TPMLP_F32) {
    const float* x = static_cast<const float*>(X);
    const float* dy = static_cast<const float*>(dY);
    float* H = at<float>(ws, w.H);
    for (int i = 0; i < n; ++i) {
      const float* Ai = static_cast<const float*>(sh->desc[i].A);
      const float* Bi = static_cast<const float*>(sh->desc[i].B);
      float* Pi = P + static_cast<size_t>(i) * T * Fs;
      float* dHi = dH + static_cast<size_t>(i) * T * Fs;
      const int t = static_cast<int>(T), d = static_cast<int>(D), fs = static_cast<int>(Fs);
      // P_i = X A_i (unless saved) ; dH_i = dY B_i^T
      if (!P_saved) TRY_CUDA(launch_simt_gemm(SimtGemm{x, D, 1, Ai, Fs, 1, Pi, Fs, t, fs, d, kSimtStore}, s));
      TRY_CUDA(launch_simt_gemm(SimtGemm{dy, D, 1, Bi, 1, D, dHi, Fs, t, fs, d, kSimtStore}, s));
    }
    // H = GeLU(P), dH <- dP = dH * GeLU'(P)
    TRY_CUDA(launch_bwd_act_f32(P, H, dH, static_cast<int64_t>(n) * T * Fs, s));
    for (int i = 0; i < n; ++i) {
      const float* Ai = static_cast<const float*>(sh->desc[i].A);
      const float* Hi = H + static_cast<size_t>(i) * T * Fs;
      const float* dPi = dH + static_cast<size_t>(i) * T * Fs;
      const int t = static_cast<int>(T), d = static_cast<int>(D), fs = static_cast<int>(Fs);
      // dB_i = H_i^T dY ; dA_i = X^T dP_i ; dX_i = dP_i A_i^T
      TRY_CUDA(launch_simt_gemm(SimtGemm{Hi, 1, Fs, dy, D, 1, static_cast<float*>(dB[i]), D, fs, d, t, kSimtStore}, s));
      TRY_CUDA(launch_simt_gemm(SimtGemm{x, 1, D, dPi, Fs, 1, static_cast<float*>(dA[i]), Fs, d, fs, t, kSimtStore}, s));
      const int epi = (!dXp && i > 0) ? kSimtAccumulate : kSimtStore;
      if (dXp || !dx_slices) {
        float* C = dXp ? dXp + static_cast<size_t>(i) * T * D : static_cast<float*>(dX);
        TRY_CUDA(launch_simt_gemm(SimtGemm{dPi, Fs, 1, Ai, 1, Fs, C, D, t, d, fs, epi}, s));
      } else {  // fused, rank slices: each slice's rows of dX straight into its buffer
        const int64_t rows = T / n;
        for (int j = 0; j < n; ++j)
          TRY_CUDA(launch_simt_gemm(SimtGemm{dPi + static_cast<size_t>(j) * rows * Fs, Fs, 1, Ai, 1, Fs,
                                             dx_slices->p[j], D, static_cast<int>(rows), d, fs, epi}, s));
      }
    }
    return finish_dx(dXp, n, T, sh, dX, tail, dx_slices, s);
  }

  // bf16: tensor-core products. X, dY, H_i and dP_i are read in place: K-major
  // where the product contracts over their columns, MN-major (64 x 64 boxes)
  // where it contracts over their rows (the token index T).
  uint16_t* H = at<uint16_t>(ws, w.H);
  uint16_t* dP = at<uint16_t>(ws, w.dP);
  CUtensorMap mX, mdY, mXmn, mdYmn;
  int major_dB = 0, major_dA = 0;  // TcMajor bits of the dB_i and dA_i products
  if ((rc = map_or_fail(&mX, X, T, D, D, tc_box_rows_a(), "X"))) return rc;
  if ((rc = map_or_fail(&mdY, dY, T, D, D, tc_box_rows_a(), "dY"))) return rc;
  if ((rc = mn_map_or_fail(&mXmn, X, T, D, D, false, &major_dA, "X (MN-major)"))) return rc;
  if ((rc = mn_map_or_fail(&mdYmn, dY, T, D, D, true, &major_dB, "dY (MN-major)"))) return rc;
  std::vector<CUtensorMap> mHmn(n), mdPmn(n), mdP(n);
  for (int i = 0; i < n; ++i) {
    uint16_t* Hi = H + static_cast<size_t>(i) * T * Fs;
    uint16_t* dPi = dP + static_cast<size_t>(i) * T * Fs;
    int mh = 0, mdp = 0;
    if ((rc = mn_map_or_fail(&mHmn[i], Hi, T, Fs, Fs, false, &mh, "H_i (MN-major)"))) return rc;
    if ((rc = mn_map_or_fail(&mdPmn[i], dPi, T, Fs, Fs, true, &mdp, "dP_i (MN-major)"))) return rc;
    if ((rc = map_or_fail(&mdP[i], dPi, T, Fs, Fs, tc_box_rows_a(), "dP_i"))) return rc;
    if (i == 0) {  // the same width for every shard, so the same map form
      major_dB |= mh;
      major_dA |= mdp;
    }
  }
  const uint64_t wl = wait_limit_ns();
  if (!P_saved && use_dual_backward(T, sh)) {
    // P_i = X A_i and dH_i = dY B_i^T in tensor memory; H_i and dP_i = dH_i *
    // GeLU'(P_i) from the epilogue.
    if ((rc = run_dual(&mX, &mdY, T, sh, H, dP, s))) return rc;
  } else {
    TcGemm g{};
    g.groups = n;
    std::vector<CUtensorMap> mo(n);
    // P_i = X A_i (recompute), fp32, unless the caller saved it.
    for (int i = 0; i < n; ++i) {
      g.map_a[i] = &mX;
      g.map_b[i] = &sh->map_At[i];
      g.out[i] = P + static_cast<size_t>(i) * T * Fs;
      if ((rc = out_map(&mo[i], g.out[i], T, Fs, Fs, "P_i"))) return rc;
      g.map_out[i] = &mo[i];
    }
    g.ldo = Fs;
    g.M = static_cast<int>(T);
    g.N = static_cast<int>(Fs);
    g.K = static_cast<int>(D);
    g.epi = kEpiF32;
    g.shared = kSharedA;  // X (then dY) feeds every shard
    g.group_m = 16;
    g.stream_out = 0;     // P is read back right away by the dH product's epilogue
    if (!P_saved) TRACED("bwd_recompute_P", s, launch_tc_gemm(g, wl, s));
    // dH_i = dY B_i^T with the activation step in its epilogue: dP_i = dH_i *
    // GeLU'(P_i) and H_i = GeLU(P_i), bf16 row-major.
    for (int i = 0; i < n; ++i) {
      g.map_a[i] = &mdY;
      g.map_b[i] = &sh->map_B[i];
      g.out[i] = dP + static_cast<size_t>(i) * T * Fs;
      g.out2[i] = H + static_cast<size_t>(i) * T * Fs;
      g.aux_p[i] = P + static_cast<size_t>(i) * T * Fs;
      g.map_out[i] = nullptr;
    }
    g.epi = kEpiBwdAct;
    TRACED("bwd_dH_act", s, launch_tc_gemm(g, wl, s));
  }
  TcGemm g{};
  g.groups = n;
  g.epi = kEpiF32;
  std::vector<CUtensorMap> mo(n);  // fp32 output maps of the current product (copied at each launch)
  // dB_i = H_i^T dY: [Fs, D], K = T; both operands MN-major.
  for (int i = 0; i < n; ++i) {
    g.map_a[i] = &mHmn[i];
    g.map_b[i] = &mdYmn;
    g.out[i] = dB[i];
    if ((rc = out_map(&mo[i], g.out[i], Fs, D, D, "dB_i"))) return rc;
    g.map_out[i] = &mo[i];
  }
  g.ldo = D;
  g.M = static_cast<int>(Fs);
  g.N = static_cast<int>(D);
  g.K = static_cast<int>(T);
  g.mn_major = major_dB;
  g.shared = kSharedB;  // dY feeds every shard
  g.group_m = 16;
  g.stream_out = 1;
  TRACED("bwd_dB", s, launch_tc_gemm(g, wl, s));
  // dA_i = X^T dP_i: [D, Fs], K = T; both operands MN-major.
  for (int i = 0; i < n; ++i) {
    g.map_a[i] = &mXmn;
    g.map_b[i] = &mdPmn[i];
    g.out[i] = dA[i];
    if ((rc = out_map(&mo[i], g.out[i], D, Fs, Fs, "dA_i"))) return rc;
  }
  g.ldo = Fs;
  g.M = static_cast<int>(D);
  g.N = static_cast<int>(Fs);
  g.mn_major = major_dA;
  g.shared = kSharedA;  // X feeds every shard
  g.group_m = 16;
  TRACED("bwd_dA", s, launch_tc_gemm(g, wl, s));
  // dX = sum_i dP_i A_i^T: [T, D], K = Fs; K-major operands.
  for (int i = 0; i < n; ++i) {
    g.map_a[i] = &mdP[i];
    g.map_b[i] = &sh->map_A[i];
    g.out[i] = dXp ? static_cast<void*>(dXp + static_cast<size_t>(i) * T * D) : dX;
    if (!dXp && dx_slices) {  // fused, rank slices: one output (and output map) per slice of T/n rows
      g.out[i] = dx_slices->p[i];
      if ((rc = out_map(&mo[i], g.out[i], T / n, D, D, "dX slice"))) return rc;
      continue;
    }
    if ((rc = out_map(&mo[i], g.out[i], T, D, D, "dX_i"))) return rc;
  }
  if (!dXp && dx_slices) g.slice_rows = T / n;
  g.ldo = D;
  g.M = static_cast<int>(T);
  g.N = static_cast<int>(D);
  g.K = static_cast<int>(Fs);
  g.mn_major = 0;
  g.chain = dXp ? 0 : 1;
  g.shared = kSharedNone;
  g.group_m = 8;
  TRACED(dXp ? "bwd_dX_partials" : "bwd_dX_fused_sum", s, launch_tc_gemm(g, wl, s));
  return finish_dx(dXp, n, T, sh, dX, tail, dx_slices, s);
}

int tpmlp_layer_norm(const void* x, int64_t T, int64_t D, tpmlp_dtype dt, float eps, void* y, tpmlp_stream_t stream) {
  if (T < 0 || D < 1) return fail(TPMLP_ERR_ARG, "T = %lld must be >= 0 and D = %lld >= 1",
                                  static_cast<long long>(T), static_cast<long long>(D));
  if (D > static_cast<int64_t>(layer_norm_max_d()))
    return fail(TPMLP_ERR_SHAPE, "D = %lld exceeds the largest supported row of %zu", static_cast<long long>(D),
                layer_norm_max_d());
  if (dt != TPMLP_F32 && dt != TPMLP_BF16) return fail(TPMLP_ERR_ARG, "unknown dtype %d", int(dt));
  int rc = check_eps(eps);
  if (rc) return rc;
  if (T == 0) return TPMLP_OK;
  if (!x || !y) return fail(TPMLP_ERR_ARG, "x and y must not be NULL");
  if (!aligned16(x) || !aligned16(y)) return fail(TPMLP_ERR_ALIGN, "x and y must be 16-byte aligned");
  if ((rc = check_device(nullptr))) return rc;
  TRACED("layer_norm", stream, launch_layer_norm(x, T, static_cast<int>(D), eps, dt == TPMLP_BF16, y, stream));
  return TPMLP_OK;
}

size_t tpmlp_block_workspace_bytes(int64_t T, const tpmlp_shards* sh, tpmlp_mode mode, int backward) {
  if (!sh || T < 1 || (mode != TPMLP_FAITHFUL && mode != TPMLP_FUSED) || backward < 0 || backward > 1) return 0;
  return plan_block(T, sh, mode, backward).total;
}

int tpmlp_block_forward(const void* x, int64_t T, const tpmlp_shards* sh, float eps, void* out, void* xn,
                        tpmlp_mode mode, void* ws, size_t ws_bytes, tpmlp_stream_t stream) {
  int rc = check_common(sh, T);
  if (rc) return rc;
  if (mode != TPMLP_FAITHFUL && mode != TPMLP_FUSED) return fail(TPMLP_ERR_ARG, "unknown mode %d", int(mode));
  if ((rc = check_eps(eps))) return rc;
  if (!x || !out || !ws) return fail(TPMLP_ERR_ARG, "x, out and workspace must not be NULL");
  if (!aligned16(x) || !aligned16(out) || !aligned16(ws) || (xn && !aligned16(xn)))
    return fail(TPMLP_ERR_ALIGN, "x, out, xn and workspace must be 16-byte aligned");
  if (sh->D > static_cast<int64_t>(layer_norm_max_d()))
    return fail(TPMLP_ERR_SHAPE, "D = %lld exceeds the largest supported row of %zu",
                static_cast<long long>(sh->D), layer_norm_max_d());
  const BlockPlan b = plan_block(T, sh, mode, 0);
  if (ws_bytes < b.total) return fail(TPMLP_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, b.total);
  if ((rc = check_handle_device(sh))) return rc;
  const bool bf16 = sh->dt == TPMLP_BF16;
  void* xnb = xn ? xn : at<char>(ws, b.xn);
  void* inner = at<char>(ws, b.inner);
  TRACED("layer_norm", stream, launch_layer_norm(x, T, static_cast<int>(sh->D), eps, bf16, xnb, stream));
  void* H = at<char>(inner, b.w.H);
  if ((rc = run_hidden(xnb, T, sh, H, stream))) return rc;
  if (mode == TPMLP_FUSED) return run_second(H, T, sh, out, 1, stream, x);
  float* Yp = at<float>(inner, b.w.Yp);
  if ((rc = run_second(H, T, sh, Yp, 0, stream))) return rc;
  TRACED("allreduce_residual", stream, launch_allreduce(Yp, sh->n, T * sh->D, static_cast<float*>(out), stream, x, bf16 ? 2 : 1));
  return TPMLP_OK;
}

int tpmlp_block_backward(const void* x, const void* dout, int64_t T, const tpmlp_shards* sh, float eps, void* dx,
                         void* const* dA, void* const* dB, tpmlp_mode mode, void* ws, size_t ws_bytes,
                         tpmlp_stream_t stream) {
  int rc = check_common(sh, T);
  if (rc) return rc;
  if (mode != TPMLP_FAITHFUL && mode != TPMLP_FUSED) return fail(TPMLP_ERR_ARG, "unknown mode %d", int(mode));
  if ((rc = check_eps(eps))) return rc;
  if (!x || !dout || !dx || !ws) return fail(TPMLP_ERR_ARG, "x, dout, dx and workspace must not be NULL");
  if (!aligned16(x) || !aligned16(dout) || !aligned16(dx) || !aligned16(ws))
    return fail(TPMLP_ERR_ALIGN, "x, dout, dx and workspace must be 16-byte aligned");
  if (sh->D > static_cast<int64_t>(layer_norm_max_d()))
    return fail(TPMLP_ERR_SHAPE, "D = %lld exceeds the largest supported row of %zu",
                static_cast<long long>(sh->D), layer_norm_max_d());
  const BlockPlan b = plan_block(T, sh, mode, 1);
  if (ws_bytes < b.total) return fail(TPMLP_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, b.total);
  if ((rc = check_handle_device(sh))) return rc;
  void* xn = at<char>(ws, b.xn);
  TRACED("layer_norm", stream, launch_layer_norm(x, T, static_cast<int>(sh->D), eps, sh->dt == TPMLP_BF16, xn, stream));
  const LnTail tail{x, dout, eps, static_cast<float*>(dx)};
  void* dxn = mode == TPMLP_FUSED ? at<char>(ws, b.dxn) : dx;  // FAITHFUL: the partials feed the tail directly
  return backward_impl(xn, dout, nullptr, T, sh, dxn, dA, dB, mode, at<char>(ws, b.inner), b.w.total, stream, &tail);
}

int tpmlp_all_gather(const void* const* slices, int n, int64_t slice_bytes, void* out, tpmlp_stream_t stream) {
  if (n < 1 || n > TPMLP_MAX_SHARDS) return fail(TPMLP_ERR_ARG, "n = %d outside 1..%d", n, TPMLP_MAX_SHARDS);
  if (slice_bytes < 0 || slice_bytes % 2 != 0)
    return fail(TPMLP_ERR_ARG, "slice_bytes = %lld must be a non-negative multiple of 2",
                static_cast<long long>(slice_bytes));
  if (slice_bytes == 0) return TPMLP_OK;
  int rc = check_slices(slices, n, "slices");
  if (rc) return rc;
  if (!out) return fail(TPMLP_ERR_ARG, "out must not be NULL");
  if (!aligned16(out)) return fail(TPMLP_ERR_ALIGN, "out must be 16-byte aligned");
  if ((rc = check_device(nullptr))) return rc;
  InSlices in{};
  for (int j = 0; j < n; ++j) in.p[j] = slices[j];
  TRACED("all_gather", stream, launch_all_gather(in, n, slice_bytes, out, stream));
  return TPMLP_OK;
}

int tpmlp_reduce_scatter(const void* Yp, int n, int64_t count, void* const* Y_slices, tpmlp_stream_t stream) {
  if (n < 1 || n > TPMLP_MAX_SHARDS) return fail(TPMLP_ERR_ARG, "n = %d outside 1..%d", n, TPMLP_MAX_SHARDS);
  if (count < 0) return fail(TPMLP_ERR_ARG, "count must be >= 0");
  if (count % n != 0)
    return fail(TPMLP_ERR_DIVISIBILITY, "count = %lld is not divisible by n = %d", static_cast<long long>(count), n);
  if (count == 0) return TPMLP_OK;
  if (!Yp) return fail(TPMLP_ERR_ARG, "Yp must not be NULL");
  if (!aligned16(Yp)) return fail(TPMLP_ERR_ALIGN, "Yp must be 16-byte aligned");
  int rc = check_slices(Y_slices, n, "Y_slices");
  if (rc) return rc;
  if ((rc = check_device(nullptr))) return rc;
  OutSlices out{};
  for (int j = 0; j < n; ++j) out.p[j] = static_cast<float*>(Y_slices[j]);
  TRACED("reduce_scatter", stream, launch_reduce_scatter(static_cast<const float*>(Yp), n, count, out, n, stream));
  return TPMLP_OK;
}

size_t tpmlp_sp_workspace_bytes(int64_t T, const tpmlp_shards* sh, tpmlp_mode mode, int backward) {
  if (!sh || T < 1 || T % sh->n != 0 || (mode != TPMLP_FAITHFUL && mode != TPMLP_FUSED) || backward < 0 ||
      backward > 1)
    return 0;
  return plan_sp(T, sh, mode, backward).total;
}

int tpmlp_forward_sp(const void* const* X_slices, int64_t T, const tpmlp_shards* sh, void* const* Y_slices,
                     tpmlp_mode mode, void* ws, size_t ws_bytes, tpmlp_stream_t stream) {
  int rc = check_common(sh, T);
  if (rc) return rc;
  if (mode != TPMLP_FAITHFUL && mode != TPMLP_FUSED) return fail(TPMLP_ERR_ARG, "unknown mode %d", int(mode));
  const int n = sh->n;
  if (n > TPMLP_MAX_SHARDS) return fail(TPMLP_ERR_UNSUPPORTED, "more than %d ranks", TPMLP_MAX_SHARDS);
  if (T % n != 0)
    return fail(TPMLP_ERR_DIVISIBILITY, "T = %lld is not divisible by n = %d", static_cast<long long>(T), n);
  if ((rc = check_slices(X_slices, n, "X_slices"))) return rc;
  if ((rc = check_slices(const_cast<const void* const*>(Y_slices), n, "Y_slices"))) return rc;
  if (!ws) return fail(TPMLP_ERR_ARG, "workspace must not be NULL");
  if (!aligned16(ws)) return fail(TPMLP_ERR_ALIGN, "workspace must be 16-byte aligned");
  const SpPlan p = plan_sp(T, sh, mode, 0);
  if (ws_bytes < p.total) return fail(TPMLP_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, p.total);
  if ((rc = check_handle_device(sh))) return rc;
  const int64_t Ts = T / n, D = sh->D;
  InSlices in{};
  OutSlices out{};
  for (int j = 0; j < n; ++j) {
    in.p[j] = X_slices[j];
    out.p[j] = static_cast<float*>(Y_slices[j]);
  }
  void* X = at<char>(ws, p.x);
  void* inner = at<char>(ws, p.inner);
  TRACED("all_gather", stream, launch_all_gather(in, n, Ts * D * static_cast<int64_t>(esize(sh->dt)), X, stream));
  void* H = at<char>(inner, p.w.H);
  if ((rc = run_hidden(X, T, sh, H, stream))) return rc;
  if (mode == TPMLP_FUSED) return run_second(H, T, sh, nullptr, 1, stream, nullptr, &out);
  float* Yp = at<float>(inner, p.w.Yp);
  if ((rc = run_second(H, T, sh, Yp, 0, stream))) return rc;
  TRACED("reduce_scatter", stream, launch_reduce_scatter(Yp, n, T * D, out, n, stream));
  return TPMLP_OK;
}

int tpmlp_backward_sp(const void* const* X_slices, const void* const* dY_slices, int64_t T, const tpmlp_shards* sh,
                      void* const* dX_slices, void* const* dA, void* const* dB, tpmlp_mode mode, void* ws,
                      size_t ws_bytes, tpmlp_stream_t stream) {
  int rc = check_common(sh, T);
  if (rc) return rc;
  if (mode != TPMLP_FAITHFUL && mode != TPMLP_FUSED) return fail(TPMLP_ERR_ARG, "unknown mode %d", int(mode));
  const int n = sh->n;
  if (n > TPMLP_MAX_SHARDS) return fail(TPMLP_ERR_UNSUPPORTED, "more than %d ranks", TPMLP_MAX_SHARDS);
  if (T % n != 0)
    return fail(TPMLP_ERR_DIVISIBILITY, "T = %lld is not divisible by n = %d", static_cast<long long>(T), n);
  if ((rc = check_slices(X_slices, n, "X_slices"))) return rc;
  if ((rc = check_slices(dY_slices, n, "dY_slices"))) return rc;
  if ((rc = check_slices(const_cast<const void* const*>(dX_slices), n, "dX_slices"))) return rc;
  if (!ws) return fail(TPMLP_ERR_ARG, "workspace must not be NULL");
  if (!aligned16(ws)) return fail(TPMLP_ERR_ALIGN, "workspace must be 16-byte aligned");
  const SpPlan p = plan_sp(T, sh, mode, 1);
  if (ws_bytes < p.total) return fail(TPMLP_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, p.total);
  if ((rc = check_handle_device(sh))) return rc;
  const int64_t slice_bytes = (T / n) * sh->D * static_cast<int64_t>(esize(sh->dt));
  InSlices in{};
  for (int j = 0; j < n; ++j) in.p[j] = X_slices[j];
  TRACED("all_gather", stream, launch_all_gather(in, n, slice_bytes, at<char>(ws, p.x), stream));
  for (int j = 0; j < n; ++j) in.p[j] = dY_slices[j];
  TRACED("all_gather", stream, launch_all_gather(in, n, slice_bytes, at<char>(ws, p.dy), stream));
  OutSlices out{};
  for (int j = 0; j < n; ++j) out.p[j] = static_cast<float*>(dX_slices[j]);
  // dX itself is never written: the partials are reduce-scattered (FAITHFUL) or
  // the product writes the slices (FUSED); slice 0 stands in for the pointer.
  return backward_impl(at<char>(ws, p.x), at<char>(ws, p.dy), nullptr, T, sh, dX_slices[0], dA, dB, mode,
                       at<char>(ws, p.inner), p.w.total, stream, nullptr, &out);
}

int tpmlp_selftest_forward_band_timeout(const void* X, int64_t T, const tpmlp_shards* sh, void* Y, tpmlp_mode mode,
                                        void* ws, size_t ws_bytes, int limit_ms, tpmlp_stream_t stream) {
  int rc = check_common(sh, T);
  if (rc) return rc;
  if (mode != TPMLP_FAITHFUL && mode != TPMLP_FUSED) return fail(TPMLP_ERR_ARG, "unknown mode %d", int(mode));
  if (!X || !Y || !ws) return fail(TPMLP_ERR_ARG, "X, Y and workspace must not be NULL");
  if (!aligned16(X) || !aligned16(Y) || !aligned16(ws))
    return fail(TPMLP_ERR_ALIGN, "X, Y and workspace must be 16-byte aligned");
  if (limit_ms < 1 || limit_ms > 10000) return fail(TPMLP_ERR_ARG, "limit_ms = %d outside 1..10000", limit_ms);
  if ((rc = check_handle_device(sh))) return rc;
  if (!use_persistent_forward(T, sh, mode))
    return fail(TPMLP_ERR_UNSUPPORTED, "this forward does not run as one persistent launch");
  const WsPlan w = plan_workspace(T, sh, mode, 0);
  if (ws_bytes < w.total) return fail(TPMLP_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, w.total);
  float* Yp = mode == TPMLP_FAITHFUL ? at<float>(ws, w.Yp) : nullptr;
  return run_forward_persistent(X, T, sh, Y, Yp, at<char>(ws, w.H), at<int>(ws, w.bands),
                                static_cast<cudaStream_t>(stream), 1, static_cast<uint64_t>(limit_ms) * 1000000ull);
}

int tpmlp_selftest_backward_withheld_fill(const void* X, const void* dY, int64_t T, const tpmlp_shards* sh, int fill,
                                          int limit_ms, void* ws, size_t ws_bytes, tpmlp_stream_t stream) {
  int rc = check_common(sh, T);
  if (rc) return rc;
  if (!X || !dY || !ws) return fail(TPMLP_ERR_ARG, "X, dY and workspace must not be NULL");
  if (!aligned16(X) || !aligned16(dY) || !aligned16(ws))
    return fail(TPMLP_ERR_ALIGN, "X, dY and workspace must be 16-byte aligned");
  if (fill < 1) return fail(TPMLP_ERR_ARG, "fill = %d must be >= 1", fill);
  if (limit_ms < 1 || limit_ms > 10000) return fail(TPMLP_ERR_ARG, "limit_ms = %d outside 1..10000", limit_ms);
  if ((rc = check_handle_device(sh))) return rc;
  if (!use_dual_backward(T, sh)) return fail(TPMLP_ERR_UNSUPPORTED, "this backward does not use the dual kernel");
  const WsPlan w = plan_workspace(T, sh, TPMLP_FUSED, 1);
  if (ws_bytes < w.total) return fail(TPMLP_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, w.total);
  const int64_t D = sh->D;
  CUtensorMap mX, mdY;
  if ((rc = map_or_fail(&mX, X, T, D, D, tc_box_rows_a(), "X"))) return rc;
  if ((rc = map_or_fail(&mdY, dY, T, D, D, tc_box_rows_a(), "dY"))) return rc;
  return run_dual(&mX, &mdY, T, sh, at<uint16_t>(ws, w.H), at<uint16_t>(ws, w.dP), static_cast<cudaStream_t>(stream),
                  fill, static_cast<uint64_t>(limit_ms) * 1000000ull);
}

int tpmlp_selftest_gemm_withheld_fill(const void* X, int64_t T, const tpmlp_shards* sh, void* H, int fill,
                                      int limit_ms, tpmlp_stream_t stream) {
  int rc = check_common(sh, T);
  if (rc) return rc;
  if (!X || !H) return fail(TPMLP_ERR_ARG, "X and H must not be NULL");
  if (!aligned16(X) || !aligned16(H)) return fail(TPMLP_ERR_ALIGN, "X and H must be 16-byte aligned");
  if (fill < 1) return fail(TPMLP_ERR_ARG, "fill = %d must be >= 1", fill);
  if (limit_ms < 1 || limit_ms > 10000) return fail(TPMLP_ERR_ARG, "limit_ms = %d outside 1..10000", limit_ms);
  if (sh->dt != TPMLP_BF16) return fail(TPMLP_ERR_UNSUPPORTED, "the tensor-core product needs bf16 shards");
  if ((rc = check_handle_device(sh))) return rc;
  return run_hidden(X, T, sh, H, stream, fill, static_cast<uint64_t>(limit_ms) * 1000000ull);
}

int tpmlp_selftest_wait_timeout(int limit_ms, tpmlp_stream_t stream) {
  if (limit_ms < 1 || limit_ms > 10000) return fail(TPMLP_ERR_ARG, "limit_ms = %d outside 1..10000", limit_ms);
  int rc = check_device(nullptr);
  if (rc) return rc;
  TRY_CUDA(launch_wait_selftest(static_cast<uint64_t>(limit_ms) * 1000000ull, stream));
  return TPMLP_OK;
}

}  // extern "C"
