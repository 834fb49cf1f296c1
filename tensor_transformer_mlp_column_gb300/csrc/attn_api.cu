// attn_api.cu — C ABI of head-split attention (include/tpmlp.h, "Head-split
// attention"): the per-rank weight handle and the forward call. Every step
// runs in kernels: the QKV projection (whose epilogue also writes V
// transposed) and the output projection on the tensor-core GEMM
// (gemm_pair.cu / gemm_tc.cu; fp32: simt.cu), the attention itself
// (attention.cu) and the sum of the output projection's partials
// (elementwise.cu); the weight set-up transposes with elementwise.cu.
#include "tpmlp.h"

#include <cmath>
#include <cstdlib>
#include <vector>

#include "internal.h"
#include "trace.h"

using namespace tpmlp;

struct tpmlp_attn_shards {
  int device = 0;
  int64_t D = 0, Dn = 0;
  int heads = 0, n = 0, dh = 0;
  tpmlp_dtype dt = TPMLP_F32;
  void* mem = nullptr;
  // Per rank i. bf16: Wqkv_i^T [3 Dn, D] (rows: the rank's columns of Wq, then
  // of Wk, then of Wv) and Wo_i^T [D, Dn]; fp32: Wqkv_i [D, 3 Dn], Wo_i [Dn, D].
  std::vector<void*> wqkv, wo;
  std::vector<CUtensorMap> map_wqkv, map_wo;  // bf16: the N x K operands of the two projections
};

namespace {

#define ATTN_TRY(expr)                                                                                  \
  do {                                                                                                  \
    cudaError_t e_ = (expr);                                                                            \
    if (e_ != cudaSuccess) return set_error(TPMLP_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_));   \
  } while (0)

// ATTN_TRY of a launch that TPMLP_TRACE=1 times as the step `phase` (trace.cu).
#define ATTN_TRACED(phase, stream, expr)    \
  do {                                      \
    TraceScope trace_scope_(phase, stream); \
    ATTN_TRY(expr);                         \
  } while (0)

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t rup(size_t x, size_t a) { return (x + a - 1) / a * a; }
size_t esz(tpmlp_dtype dt) { return dt == TPMLP_BF16 ? 2 : 4; }
int64_t rup8(int64_t x) { return (x + 7) / 8 * 8; }

uint64_t attn_wait_ns() {
  const char* s = getenv("TPMLP_WAIT_LIMIT_MS");
  long ms = s ? atol(s) : 0;
  if (ms <= 0 || ms > 600000) ms = 4000;
  return static_cast<uint64_t>(ms) * 1000000ull;
}

int current_sm103(int* dev_out) {
  int dev = -1, major = 0, minor = 0;
  ATTN_TRY(cudaGetDevice(&dev));
  ATTN_TRY(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
  ATTN_TRY(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
  if (major != 10 || minor != 3)
    return set_error(TPMLP_ERR_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a (GB300)", dev, major,
                     minor);
  if (dev_out) *dev_out = dev;
  return TPMLP_OK;
}

// Workspace: QKV [n][T][3 Dn], V^T [n][Dn][T8] (bf16), O [n][T][Dn], and in
// FAITHFUL mode the output projection's partials Yp [n][T][D] fp32.
struct AttnPlan {
  size_t qkv = 0, vt = 0, o = 0, yp = 0, total = 0;
};

AttnPlan plan_attn(int64_t T, const tpmlp_attn_shards* sh, int mode_or_heads_only) {
  AttnPlan p;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = rup(off + bytes, 256);
    return at;
  };
  const size_t n = sh->n, Dn = sh->Dn, D = sh->D, t = T, es = esz(sh->dt);
  p.qkv = take(n * t * 3 * Dn * es);
  if (sh->dt == TPMLP_BF16) p.vt = take(n * Dn * rup8(T) * 2);
  if (mode_or_heads_only >= 0) {  // forward: O and, FAITHFUL, the partials
    p.o = take(n * t * Dn * es);
    if (mode_or_heads_only == TPMLP_FAITHFUL) p.yp = take(n * t * D * 4);
  }
  p.total = off;
  return p;
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

int check_attn(const tpmlp_attn_shards* sh, int64_t batch, int64_t seq) {
  if (!sh) return set_error(TPMLP_ERR_ARG, "attention shards handle is NULL");
  if (batch < 1 || seq < 1) return set_error(TPMLP_ERR_ARG, "batch and seq must be >= 1");
  if (sh->dt == TPMLP_F32 && seq > 8192)
    return set_error(TPMLP_ERR_SHAPE, "fp32 attention supports seq up to 8192 (seq = %lld)", static_cast<long long>(seq));
  if (batch * seq > (int64_t(1) << 30)) return set_error(TPMLP_ERR_ARG, "batch * seq is too large");
  if (sh->dt == TPMLP_BF16 && seq % 8 != 0)
    return set_error(TPMLP_ERR_SHAPE, "bf16 attention needs seq %% 8 == 0 (seq = %lld)", static_cast<long long>(seq));
  int dev = -1;
  int rc = current_sm103(&dev);
  if (rc) return rc;
  if (dev != sh->device)
    return set_error(TPMLP_ERR_DEVICE, "attention shards live on device %d but device %d is current", sh->device, dev);
  return TPMLP_OK;
}

// QKV_i = X Wqkv_i, V_i^T, O_i = attention of rank i's heads; O [n][T][Dn].
int run_heads(const void* X, int64_t batch, int64_t seq, const tpmlp_attn_shards* sh, void* O, void* ws,
              const AttnPlan& pl, cudaStream_t s) {
  const int64_t T = batch * seq, D = sh->D, Dn = sh->Dn;
  const int n = sh->n;
  void* qkv = at<char>(ws, pl.qkv);
  if (sh->dt == TPMLP_F32) {
    for (int i = 0; i < n; ++i) {
      SimtGemm g{static_cast<const float*>(X), D, 1, static_cast<const float*>(sh->wqkv[i]), 3 * Dn, 1,
                 static_cast<float*>(qkv) + static_cast<size_t>(i) * T * 3 * Dn, 3 * Dn, static_cast<int>(T),
                 static_cast<int>(3 * Dn), static_cast<int>(D), kSimtStore};
      ATTN_TRY(launch_simt_gemm(g, s));
    }
    ATTN_TRY(launch_attention_f32(static_cast<const float*>(qkv), T, n, static_cast<int>(Dn), sh->dh,
                                  sh->heads / n, static_cast<int>(batch), static_cast<int>(seq),
                                  static_cast<float*>(O), s));
    return TPMLP_OK;
  }
  // bf16: the QKV projection of every rank in one grouped tensor-core product
  // (X shared by all ranks) whose epilogue writes Q, K row-major and V
  // transposed, then the attention kernel.
  CUtensorMap mx;
  if (!make_operand_map(&mx, X, T, D, D, tc_box_rows_a()))
    return set_error(TPMLP_ERR_CUDA, "cuTensorMapEncodeTiled rejected the map of X");
  TcGemm g{};
  g.groups = n;
  const int64_t T8 = rup8(T);
  for (int i = 0; i < n; ++i) {
    g.map_a[i] = &mx;
    g.map_b[i] = &sh->map_wqkv[i];
    g.out[i] = at<uint16_t>(qkv, 0) + static_cast<size_t>(i) * T * 3 * Dn;
    g.aux_ht[i] = at<uint16_t>(ws, pl.vt) + static_cast<size_t>(i) * Dn * T8;  // V_i^T [Dn, T8] from the epilogue
  }
  g.vt_col0 = static_cast<int>(2 * Dn);
  g.ldt = T8;
  g.ldo = 3 * Dn;
  g.M = static_cast<int>(T);
  g.N = static_cast<int>(3 * Dn);
  g.K = static_cast<int>(D);
  g.epi = kEpiBf16;
  g.shared = kSharedA;
  g.group_m = 16;
  ATTN_TRACED("attn_qkv", s, launch_tc_gemm(g, attn_wait_ns(), s));
  std::vector<CUtensorMap> mq(n), mv(n);
  AttnLaunch a{};
  for (int i = 0; i < n; ++i) {
    uint16_t* qkv_i = at<uint16_t>(qkv, 0) + static_cast<size_t>(i) * T * 3 * Dn;
    uint16_t* vt_i = at<uint16_t>(ws, pl.vt) + static_cast<size_t>(i) * Dn * T8;
    if (!make_operand_map(&mq[i], qkv_i, T, 3 * Dn, 3 * Dn, 128) || !make_operand_map(&mv[i], vt_i, Dn, T, T8, 64))
      return set_error(TPMLP_ERR_CUDA, "cuTensorMapEncodeTiled rejected a map of rank %d's Q, K or V^T", i);
    a.map_qkv[i] = &mq[i];
    a.map_vt[i] = &mv[i];
    a.out[i] = static_cast<uint16_t*>(O) + static_cast<size_t>(i) * T * Dn;
  }
  a.n = n;
  a.batch = static_cast<int>(batch);
  a.seq = static_cast<int>(seq);
  a.Dn = static_cast<int>(Dn);
  a.local_heads = sh->heads / n;
  a.wait_ns = attn_wait_ns();
  a.status = device_status_word();
  if (!a.status) return set_error(TPMLP_ERR_CUDA, "the device status word is not available");
  ATTN_TRACED("attn_core", s, launch_attention_tc(a, s));
  return TPMLP_OK;
}

}  // namespace

extern "C" {

int tpmlp_attn_shard(const void* Wq, const void* Wk, const void* Wv, const void* Wo, int64_t D, int heads, int n,
                     tpmlp_dtype dt, tpmlp_stream_t stream, tpmlp_attn_shards** out) {
  if (!out) return set_error(TPMLP_ERR_ARG, "out must not be NULL");
  *out = nullptr;
  if (!Wq || !Wk || !Wv || !Wo) return set_error(TPMLP_ERR_ARG, "Wq, Wk, Wv and Wo must not be NULL");
  if (dt != TPMLP_F32 && dt != TPMLP_BF16) return set_error(TPMLP_ERR_ARG, "unknown dtype %d", int(dt));
  if (D < 1 || heads < 1 || n < 1) return set_error(TPMLP_ERR_ARG, "D, heads and n must be >= 1");
  if (D % heads != 0 || heads % n != 0)
    return set_error(TPMLP_ERR_DIVISIBILITY, "D = %lld must be divisible by heads = %d and heads by n = %d",
                     static_cast<long long>(D), heads, n);
  if (n > TPMLP_MAX_SHARDS) return set_error(TPMLP_ERR_UNSUPPORTED, "more than %d ranks", TPMLP_MAX_SHARDS);
  const int dh = static_cast<int>(D / heads);
  if (dt == TPMLP_BF16 && dh != 64)
    return set_error(TPMLP_ERR_UNSUPPORTED, "bf16 attention is built for a head size of 64 (got %d)", dh);
  if (dt == TPMLP_F32 && dh > 128)
    return set_error(TPMLP_ERR_UNSUPPORTED, "fp32 attention supports head sizes up to 128 (got %d)", dh);
  if (!al16(Wq) || !al16(Wk) || !al16(Wv) || !al16(Wo))
    return set_error(TPMLP_ERR_ALIGN, "Wq, Wk, Wv and Wo must be 16-byte aligned");
  int dev = -1;
  int rc = current_sm103(&dev);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto* sh = new tpmlp_attn_shards;
  sh->device = dev;
  sh->D = D;
  sh->Dn = D / n;
  sh->heads = heads;
  sh->n = n;
  sh->dh = dh;
  sh->dt = dt;
  const size_t es = esz(dt), Dn = static_cast<size_t>(D / n);
  const size_t blk_qkv = rup(static_cast<size_t>(D) * 3 * Dn * es, 256), blk_o = rup(static_cast<size_t>(D) * Dn * es, 256);
  if (cudaMalloc(&sh->mem, n * (blk_qkv + blk_o)) != cudaSuccess) {
    delete sh;
    return set_error(TPMLP_ERR_CUDA, "cudaMalloc of %zu bytes for the attention shards failed", n * (blk_qkv + blk_o));
  }
  const void* W3[3] = {Wq, Wk, Wv};
  for (int i = 0; i < n; ++i) {
    char* base = static_cast<char*>(sh->mem) + i * (blk_qkv + blk_o);
    sh->wqkv.push_back(base);
    sh->wo.push_back(base + blk_qkv);
    cudaError_t e = cudaSuccess;
    if (dt == TPMLP_BF16) {
      // Wqkv_i^T rows [k Dn, (k+1) Dn) = (W_k[:, i Dn : (i+1) Dn])^T; Wo_i^T = (Wo[i Dn : (i+1) Dn, :])^T.
      for (int k = 0; k < 3 && e == cudaSuccess; ++k)
        e = launch_transpose_u16(static_cast<const uint16_t*>(W3[k]) + i * Dn, D, static_cast<int64_t>(Dn), D,
                                 static_cast<uint16_t*>(sh->wqkv[i]) + k * Dn * D, D, s);
      if (e == cudaSuccess)
        e = launch_transpose_u16(static_cast<const uint16_t*>(Wo) + i * Dn * D, static_cast<int64_t>(Dn), D, D,
                                 sh->wo[i], static_cast<int64_t>(Dn), s);
    } else {
      // Wqkv_i = [Wq_i | Wk_i | Wv_i] [D, 3 Dn]; Wo_i = rows i Dn .. of Wo.
      for (int k = 0; k < 3 && e == cudaSuccess; ++k)
        e = cudaMemcpy2DAsync(static_cast<float*>(sh->wqkv[i]) + k * Dn, 3 * Dn * 4,
                              static_cast<const float*>(W3[k]) + i * Dn, D * 4, Dn * 4, D, cudaMemcpyDeviceToDevice, s);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(sh->wo[i], static_cast<const float*>(Wo) + i * Dn * D, Dn * D * 4,
                            cudaMemcpyDeviceToDevice, s);
    }
    if (e != cudaSuccess) {
      cudaFree(sh->mem);
      delete sh;
      return set_error(TPMLP_ERR_CUDA, "building rank %d's weights: %s", i, cudaGetErrorString(e));
    }
  }
  if (dt == TPMLP_BF16) {
    sh->map_wqkv.resize(n);
    sh->map_wo.resize(n);
    for (int i = 0; i < n; ++i) {
      if (!make_operand_map(&sh->map_wqkv[i], sh->wqkv[i], 3 * static_cast<int64_t>(Dn), D, D,
                            tc_box_rows_b(static_cast<int>(3 * Dn))) ||
          !make_operand_map(&sh->map_wo[i], sh->wo[i], D, static_cast<int64_t>(Dn), static_cast<int64_t>(Dn),
                            tc_box_rows_b(static_cast<int>(D)))) {
        cudaFree(sh->mem);
        delete sh;
        return set_error(TPMLP_ERR_CUDA, "cuTensorMapEncodeTiled rejected rank %d's weight maps", i);
      }
    }
  }
  *out = sh;
  return TPMLP_OK;
}

int tpmlp_attn_shard_get(const tpmlp_attn_shards* sh, int i, const void** Wqkv_i, const void** Wo_i) {
  if (!sh || i < 0 || i >= sh->n || !Wqkv_i || !Wo_i) return set_error(TPMLP_ERR_ARG, "bad handle, index or pointer");
  *Wqkv_i = sh->wqkv[i];
  *Wo_i = sh->wo[i];
  return TPMLP_OK;
}

void tpmlp_attn_shards_free(tpmlp_attn_shards* sh) {
  if (!sh) return;
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != sh->device) cudaSetDevice(sh->device);
  cudaDeviceSynchronize();
  if (sh->mem) cudaFree(sh->mem);
  if (prev >= 0 && prev != sh->device) cudaSetDevice(prev);
  delete sh;
}

size_t tpmlp_attn_workspace_bytes(int64_t batch, int64_t seq, const tpmlp_attn_shards* sh, int mode) {
  if (!sh || batch < 1 || seq < 1 || mode < -1 || mode > 1) return 0;
  return plan_attn(batch * seq, sh, mode).total;
}

int tpmlp_attn_heads(const void* X, int64_t batch, int64_t seq, const tpmlp_attn_shards* sh, void* O, void* ws,
                     size_t ws_bytes, tpmlp_stream_t stream) {
  int rc = check_attn(sh, batch, seq);
  if (rc) return rc;
  if (!X || !O || !ws) return set_error(TPMLP_ERR_ARG, "X, O and workspace must not be NULL");
  if (!al16(X) || !al16(O) || !al16(ws)) return set_error(TPMLP_ERR_ALIGN, "X, O and workspace must be 16-byte aligned");
  const AttnPlan pl = plan_attn(batch * seq, sh, -1);
  if (ws_bytes < pl.total)
    return set_error(TPMLP_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, pl.total);
  return run_heads(X, batch, seq, sh, O, ws, pl, static_cast<cudaStream_t>(stream));
}

int tpmlp_attn_forward(const void* X, int64_t batch, int64_t seq, const tpmlp_attn_shards* sh, void* Y,
                       tpmlp_mode mode, void* ws, size_t ws_bytes, tpmlp_stream_t stream) {
  int rc = check_attn(sh, batch, seq);
  if (rc) return rc;
  if (mode != TPMLP_FAITHFUL && mode != TPMLP_FUSED) return set_error(TPMLP_ERR_ARG, "unknown mode %d", int(mode));
  if (!X || !Y || !ws) return set_error(TPMLP_ERR_ARG, "X, Y and workspace must not be NULL");
  if (!al16(X) || !al16(Y) || !al16(ws)) return set_error(TPMLP_ERR_ALIGN, "X, Y and workspace must be 16-byte aligned");
  const int64_t T = batch * seq, D = sh->D, Dn = sh->Dn;
  const int n = sh->n;
  const AttnPlan pl = plan_attn(T, sh, mode);
  if (ws_bytes < pl.total)
    return set_error(TPMLP_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, pl.total);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* O = at<char>(ws, pl.o);
  if ((rc = run_heads(X, batch, seq, sh, O, ws, pl, s))) return rc;
  float* Yp = mode == TPMLP_FAITHFUL ? at<float>(ws, pl.yp) : nullptr;
  // Output projection, row-parallel: Y_i = O_i Wo_i (partials) or their
  // on-chip shard-ordered sum; the partials then go through the MLP's reduce.
  if (sh->dt == TPMLP_F32) {
    for (int i = 0; i < n; ++i) {
      float* C = Yp ? Yp + static_cast<size_t>(i) * T * D : static_cast<float*>(Y);
      SimtGemm g{static_cast<const float*>(O) + static_cast<size_t>(i) * T * Dn, Dn, 1,
                 static_cast<const float*>(sh->wo[i]), D, 1, C, D, static_cast<int>(T), static_cast<int>(D),
                 static_cast<int>(Dn), (!Yp && i > 0) ? kSimtAccumulate : kSimtStore};
      ATTN_TRY(launch_simt_gemm(g, s));
    }
  } else {
    std::vector<CUtensorMap> mo(n), mout(n);
    TcGemm g{};
    g.groups = n;
    for (int i = 0; i < n; ++i) {
      if (!make_operand_map(&mo[i], static_cast<uint16_t*>(O) + static_cast<size_t>(i) * T * Dn, T, Dn, Dn,
                            tc_box_rows_a()))
        return set_error(TPMLP_ERR_CUDA, "cuTensorMapEncodeTiled rejected the map of O_%d", i);
      g.map_a[i] = &mo[i];
      g.map_b[i] = &sh->map_wo[i];
      g.out[i] = Yp ? static_cast<void*>(Yp + static_cast<size_t>(i) * T * D) : Y;
      if (!make_output_map_f32(&mout[i], g.out[i], T, D, D))
        return set_error(TPMLP_ERR_CUDA, "cuTensorMapEncodeTiled rejected the output map of Y_%d", i);
      g.map_out[i] = &mout[i];
    }
    g.ldo = D;
    g.M = static_cast<int>(T);
    g.N = static_cast<int>(D);
    g.K = static_cast<int>(Dn);
    g.chain = Yp ? 0 : 1;
    g.epi = kEpiF32;
    g.group_m = 8;
    g.stream_out = 1;
    ATTN_TRACED("attn_out_proj", s, launch_tc_gemm(g, attn_wait_ns(), s));
  }
  if (Yp) ATTN_TRACED("allreduce", s, launch_allreduce(Yp, n, T * D, static_cast<float*>(Y), s));
  return TPMLP_OK;
}

}  // extern "C"
