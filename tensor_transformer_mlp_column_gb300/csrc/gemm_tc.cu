// gemm_tc.cu — tensor-core GEMM entry: the launcher that picks a kernel for
// each product, the single-CTA tcgen05 kernel for small products, the TMA map
// helpers, and the device status word with its self test.
//
// Single-CTA kernel: one CTA per SM loops over output tiles of 128 x BN
// (BN = 64, 128 or 256):
//   warp 0, lane 0 : TMA producer — fills a STAGES-deep ring of shared-memory
//                    stages (A 128 x 64, B BN x 64, 128-byte swizzle)
//   warp 1         : allocates TMEM; lane 0 issues tcgen05.mma (M=128, N=BN,
//                    K=16 per instruction) into one of two TMEM accumulators
//   warps 2..5     : epilogue — tcgen05.ld the accumulator (warp w reads TMEM
//                    lanes 32*(w%4)..+31 = tile rows), apply the output
//                    treatment and store to global memory
// The two accumulators let the epilogue of tile j overlap the mainloop of
// tile j+1. Every mbarrier wait is bounded; on a timeout the CTA raises an
// abort flag, all roles leave their loops, in-flight copies and MMAs are
// drained and TMEM is freed before the CTA exits.
#include "gemm_common.cuh"

#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <cstring>

namespace tpmlp {

// Per-device status word: a kernel whose bounded wait ran out of time stores
// the wait's site code here. Read and cleared by read_and_clear_status().
__device__ int g_status = 0;

namespace {

// A stage holds KSUB consecutive 64-column K blocks: two for 128-column
// tiles (three stages of 64 KB, half the barrier round trips per MMA) and for
// 64-column tiles (four stages of 48 KB), one for 256-column tiles (four
// stages of 48 KB).
template <int BN>
struct Cfg {
  static constexpr int KSUB = BN <= 128 ? 2 : 1;
  static constexpr int STAGES = BN == 128 ? 3 : 4;
  static constexpr uint32_t A_SUB = BM * BK * 2;  // one K block of the M x K operand
  static constexpr uint32_t B_SUB = BN * BK * 2;  // one K block of the N x K operand
  static constexpr uint32_t A_BYTES = KSUB * A_SUB;
  static constexpr uint32_t B_BYTES = KSUB * B_SUB;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TMEM_COLS = 2 * BN;  // two accumulators
  static constexpr size_t SMEM = 1024 /*alignment slack*/ + size_t(STAGES) * STAGE_BYTES + 256 /*barriers*/;
};

template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ KParams p) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full + b, 1);
      mbar_init(acc_empty + b, 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    const int ng = p.groups;
    for (int g = 0; g < ng; ++g) {
      tma_prefetch_desc(&p.map_a[g]);
      tma_prefetch_desc(&p.map_b[g]);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // Set-up done: from here on global memory is read and written, so wait for
  // the previous kernel of the stream, and let the next one start its set-up.
  pdl_wait();
  pdl_launch_dependents();
  const WaitGuard guard{abort_flag, p.wait_ns, p.status};
  const int kb_per_tile = p.chain ? p.groups * p.k_blocks : p.k_blocks;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, parity_bits = 0;
      int fill = 0;
      bool ok = true;
      const uint64_t pol_a = l2_policy(p.load_hint & 3), pol_b = l2_policy((p.load_hint >> 2) & 3);
      for (int tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
        int g, mb, nb;
        decode_tile(p, tile, g, mb, nb);
        if (!tile_ok(p, g, mb, nb)) continue;
        int gg = g, kk = 0;  // group and K block of the next load (chain mode walks the groups in order)
        for (int kb = 0; kb < kb_per_tile; kb += C::KSUB) {
          if (!wait_bounded(empty + stage, phase ^ 1u, guard, kSiteProducer)) {
            ok = false;
            break;
          }
          const int nsub = kb_per_tile - kb < C::KSUB ? kb_per_tile - kb : C::KSUB;  // K blocks in this stage
          ++fill;
          // Inner (x) coordinates of this stage's loads must be 16-byte aligned.
          if (!TPMLP_DCHECK((kk * BK) % 8 == 0 && (mb * BM) % 64 == 0 && (nb * BN) % 64 == 0, p.status, kChkTmaX)) {
            ok = false;
            *abort_flag = 1;
            break;
          }
          if (fill != p.inject) {
            mbar_arrive_expect_tx(full + stage, nsub * (C::A_SUB + C::B_SUB));
            for (int u = 0; u < nsub; ++u) {
              uint8_t* da = sA + stage * C::A_BYTES + u * C::A_SUB;
              uint8_t* db = sB + stage * C::B_BYTES + u * C::B_SUB;
              // MN-major operands ([K][M] tensors): 64-wide chunks of 64 K rows,
              // two per box of a 3-D map or one per box of a 2-D one.
              if (p.mn_major & kMnA3d) {
                tma_load_3d_hint(da, &p.map_a[gg], 0, kk * BK, mb * BM / 64, full + stage, pol_a);
              } else if (p.mn_major & kMnA) {
                for (int c = 0; c < BM / 64; ++c)
                  tma_load_2d_hint(da + c * kMnChunkBytes, &p.map_a[gg], mb * BM + 64 * c, kk * BK, full + stage,
                                   pol_a);
              } else {
                tma_load_2d_hint(da, &p.map_a[gg], kk * BK, mb * BM, full + stage, pol_a);
              }
              if (p.mn_major & kMnB3d) {
                for (int c = 0; c < BN / 128; ++c)
                  tma_load_3d_hint(db + c * 2 * kMnChunkBytes, &p.map_b[gg], 0, kk * BK, (nb * BN + 128 * c) / 64,
                                   full + stage, pol_b);
              } else if (p.mn_major & kMnB) {
                for (int c = 0; c < BN / 64; ++c)
                  tma_load_2d_hint(db + c * kMnChunkBytes, &p.map_b[gg], nb * BN + 64 * c, kk * BK, full + stage,
                                   pol_b);
              } else {
                tma_load_2d_hint(db, &p.map_b[gg], kk * BK, nb * BN, full + stage, pol_b);
              }
              if (++kk == p.k_blocks) {
                kk = 0;
                ++gg;
              }
            }
            issued |= 1u << stage;
            parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
          } else {
            for (int u = 0; u < nsub; ++u)  // the withheld fill still advances the K position
              if (++kk == p.k_blocks) {
                kk = 0;
                ++gg;
              }
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Leave no copy in flight into this CTA's shared memory.
        for (int s = 0; s < C::STAGES; ++s)
          if (issued >> s & 1u) wait_drain(full + s, (parity_bits >> s) & 1u, p.wait_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      const bool a_mn = (p.mn_major & kMnA) != 0, b_mn = (p.mn_major & kMnB) != 0;
      const uint32_t idesc = idesc_bf16_f32(BM, BN, a_mn, b_mn);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
        if constexpr (kDebugBuild) {
          int g, mb, nb;
          decode_tile(p, tile, g, mb, nb);
          if (!tile_ok(p, g, mb, nb)) continue;
        }
        if (!wait_bounded(acc_empty + acc, acc_phase ^ 1u, guard, kSiteMmaAcc)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < kb_per_tile; kb += C::KSUB) {
          if (!wait_bounded(full + stage, phase, guard, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const int nsub = kb_per_tile - kb < C::KSUB ? kb_per_tile - kb : C::KSUB;
          for (int u = 0; u < nsub; ++u) {
            const uint32_t a0 = smem_addr(sA + stage * C::A_BYTES + u * C::A_SUB);
            const uint32_t b0 = smem_addr(sB + stage * C::B_BYTES + u * C::B_SUB);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              tc_mma_bf16(d_tmem, operand_desc(a0, k, a_mn), operand_desc(b0, k, b_mn), idesc,
                          (kb | u | k) != 0 ? 1u : 0u);
            }
          }
          tc_commit(empty + stage);  // frees the stage once these MMAs have read it
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(acc_full + acc);  // accumulator complete
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        // Let every MMA already issued finish before TMEM is released.
        tc_commit(drain);
        wait_drain(drain, 0, p.wait_ns);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5)
    const int quarter = warp & 3;  // the TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x) {
      int g, mb, nb;
      decode_tile(p, tile, g, mb, nb);
      if (!tile_ok(p, g, mb, nb)) continue;
      bool ok = wait_bounded(acc_full + acc, acc_phase, guard, kSiteEpilogue);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after_sync();
      const int64_t m = int64_t(mb) * BM + row;
      const bool row_ok = m < p.M;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        float v[32];
        const int n0 = nb * BN + c;
        uint4 res[4];
        const bool with_res = EPI == kEpiF32 && p.resid != nullptr && row_ok && n0 < p.N;
        if (with_res) load_residual(p, m, n0, res);
        __syncwarp();  // tcgen05.ld is warp-collective
        tmem_ld_32cols(t_row + static_cast<uint32_t>(c), v);
        if (with_res) add_residual(res, v);
        if (c + 32 == BN) {
          // The accumulator may be overwritten now; the arrival orders only
          // these completed TMEM reads, so it is relaxed.
          tc_fence_before_sync();
          mbar_arrive_relaxed(acc_empty + acc);
        }
        if (!row_ok || n0 >= p.N) continue;
        epilogue_store<EPI>(p, g, m, n0, v);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int BN, int EPI>
cudaError_t launch_single(const KParams& kp, cudaStream_t s) {
  using C = Cfg<BN>;
  auto kern = tc_gemm_kernel<BN, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::SMEM));
  if (e != cudaSuccess) return e;
  const int grid = kp.tiles < num_sms() ? kp.tiles : num_sms();
  e = launch_pdl(kern, dim3(grid), dim3(kThreads), C::SMEM, s, kp);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int BN>
cudaError_t launch_single_epi(const KParams& kp, int epi, cudaStream_t s) {
  switch (epi) {
    case kEpiGeluBf16:
      return launch_single<BN, kEpiGeluBf16>(kp, s);
    case kEpiF32:
      return launch_single<BN, kEpiF32>(kp, s);
    case kEpiBwdAct:
      return launch_single<BN, kEpiBwdAct>(kp, s);
    case kEpiGeluSaveP:
      return launch_single<BN, kEpiGeluSaveP>(kp, s);
    case kEpiBf16:
      return launch_single<BN, kEpiBf16>(kp, s);
    default:
      return cudaErrorInvalidValue;
  }
}

// Waits on a barrier that expects one arrival that never comes; the bounded
// wait gives up after limit_ns and records kSiteSelftest.
__global__ void wait_selftest_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitGuard g{&abort_flag, limit_ns, &g_status};
    wait_bounded(&bar, 0, g, kSiteSelftest);
  }
}

// The debug build's check in isolation: thread 0 writes element `index` of a
// 32-element shared array only if the check passes. In the normal build the
// kernel does nothing (and the C ABI never launches it).
__global__ void bounds_selftest_kernel(int index, int* status) {
#ifdef TPMLP_DEBUG
  __shared__ int buf[32];
  buf[threadIdx.x] = 0;
  __syncthreads();
  if (threadIdx.x == 0 && TPMLP_DCHECK(index >= 0 && index < 32, status, kChkSelftest)) buf[index] = 1;
  __syncthreads();
  if (buf[threadIdx.x] > 1) atomicAdd(status, 0);  // keeps the store from being removed
#else
  (void)index;
  (void)status;
#endif
}

int env_int(const char* name, int dflt) {
  const char* e = getenv(name);
  return e && *e ? atoi(e) : dflt;
}

// Kernel family for the bf16 products, read once per process: 1 = CTA pairs
// for products with enough 256 x 256 tiles, 0 = single CTAs only.
// TPMLP_TC_KERNEL overrides the default for comparisons.
int kernel_family() {
  static const int v = [] {
    const int f = env_int("TPMLP_TC_KERNEL", 1);
    return f < 0 || f > 1 ? 1 : f;
  }();
  return v;
}

// Device address of g_status on the current device.
int* status_word() {
  static std::atomic<int*> cached[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  int* w = cached[dev].load(std::memory_order_relaxed);
  if (!w) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status) == cudaSuccess) {
      w = static_cast<int*>(ptr);
      cached[dev].store(w, std::memory_order_relaxed);
    }
  }
  return w;
}

}  // namespace

int* device_status_word() { return status_word(); }

bool tc_pairs_enabled() { return kernel_family() >= 1; }

bool pdl_enabled() {
  static const bool v = env_int("TPMLP_PDL", 1) != 0;
  return v;
}

cudaError_t launch_bounds_selftest(int index, cudaStream_t s) {
  if (!kDebugBuild) return cudaErrorNotSupported;
  int* st = status_word();
  if (!st) return cudaErrorInvalidSymbol;
  bounds_selftest_kernel<<<1, 32, 0, s>>>(index, st);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t read_and_clear_status(int* value, cudaStream_t s) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(value, g_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(s);  // `zero` and `value` are host stack memory
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

// Box heights of the operand maps: the M x K operand in 128-row boxes; the
// N x K operand in 128-row boxes (each CTA of a pair loads half of the 256 N
// rows), or BN rows for the single-CTA kernel when it is the only family in
// use.
int tc_box_rows_a() { return 128; }
int tc_box_rows_b(int N) {
  if (kernel_family() >= 1) return 128;
  return N <= 128 ? 128 : 256;
}

// A 2-D row-major tensor [rows, cols] with a row pitch of pitch_bytes, boxes
// of box_cols x box_rows elements, 128-byte swizzle.
static bool encode_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, int64_t rows, int64_t cols,
                      int64_t pitch_bytes, int box_cols, int box_rows) {
  static const PFN_cuTensorMapEncodeTiled_v12000 encode = [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      fn = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }();
  if (!encode) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_operand_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t pitch_elems,
                      int box_rows) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rows, cols, pitch_elems * 2, BK, box_rows);
}

bool make_operand_map_mn3d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t pitch_elems) {
  if (cols % 64 != 0 || cols > pitch_elems) return false;
  static const PFN_cuTensorMapEncodeTiled_v12000 encode = [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      fn = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }();
  if (!encode) return false;
  // Element (i, k, c) = base[k * pitch + 64 c + i]: the row-major [rows][cols]
  // tensor seen as cols / 64 chunks of 64 columns.
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(pitch_elems * 2), 128};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BK), 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_output_map_f32(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t pitch_elems) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, rows, cols, pitch_elems * 4, 32, 32);
}

bool make_output_map_bf16(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t pitch_elems) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rows, cols, pitch_elems * 2, 64, 32);
}

cudaError_t launch_tc_gemm(const TcGemm& g, uint64_t wait_ns, cudaStream_t s) {
  KParams kp;
  memset(&kp, 0, sizeof(kp));
  for (int i = 0; i < g.groups; ++i) {
    kp.map_a[i] = *g.map_a[i];
    kp.map_b[i] = *g.map_b[i];
    kp.out[i] = g.out[i];
    kp.out2[i] = g.out2[i];
    kp.aux_p[i] = g.aux_p[i];
    kp.aux_ht[i] = g.aux_ht[i];
    if (g.map_out[i]) kp.map_out[i] = *g.map_out[i];
  }
  // CTA pairs with 256 x 256 tiles, unless the product has too few
  // of those tiles to occupy a quarter of the SMs: then single CTAs with
  // 128 x 128 tiles (the N x K boxes that pair mode encodes) spread it over
  // four times as many SMs.
  const int family = kernel_family();
  const int pair_tiles = ((g.M + 255) / 256) * ((g.N + 255) / 256) * (g.chain ? 1 : g.groups);
  const bool pair = family >= 1 && pair_tiles >= num_sms() / 4;
  int BN = pair ? 256 : tc_box_rows_b(g.N);
  // A single-CTA product that is read from L2 at the SM's load rate (128 x 128
  // tiles load 32 KB per 64-deep K block, 256 MMA cycles of work) moves to
  // 128 x 64 tiles (24 KB per 128 MMA cycles) when their twice as many tiles
  // still fit in one round over the SMs: a quarter less to load per SM, on
  // twice as many SMs. Needs the 64-row maps of the N x K operand.
  bool narrow_maps = g.groups > 0;
  for (int i = 0; i < g.groups; ++i) narrow_maps = narrow_maps && g.map_b_narrow[i] != nullptr;
  if (!pair && BN == 128 && narrow_maps && env_int("TPMLP_NARROW", 1) != 0) {
    const int64_t units = int64_t((g.M + BM - 1) / BM) * (g.chain ? 1 : g.groups);
    const int64_t t128 = units * ((g.N + 127) / 128), t64 = units * ((g.N + 63) / 64);
    const int64_t sms = num_sms();
    if ((t64 + sms - 1) / sms <= (t128 + sms - 1) / sms) BN = 64;
  }
  const int TM = pair ? 256 : BM;
  if (BN == 64)
    for (int i = 0; i < g.groups; ++i) kp.map_b[i] = *g.map_b_narrow[i];
  kp.ldo = g.ldo;
  kp.ldt = g.ldt;
  kp.M = g.M;
  kp.N = g.N;
  kp.groups = g.groups;
  kp.chain = g.chain;
  kp.m_blocks = (g.M + TM - 1) / TM;
  kp.n_blocks = (g.N + BN - 1) / BN;
  kp.k_blocks = (g.K + BK - 1) / BK;
  kp.tiles = kp.m_blocks * kp.n_blocks * (g.chain ? 1 : g.groups);
  kp.wait_ns = wait_ns;
  kp.status = status_word();
  kp.inject = g.inject;
  kp.group_m = env_int("TPMLP_GROUP_M", g.group_m);
  kp.shared = g.shared;
  kp.stream_out = env_int("TPMLP_STREAM_OUT", g.stream_out);
  // Operand tiles are read by several CTAs (the tiles of a band share them):
  // loaded with the evict-last L2 priority so that the output stream does
  // not push them out first (TPMLP_LOAD_HINT=0 loads them with normal priority).
  kp.load_hint = env_int("TPMLP_LOAD_HINT", 1 | (1 << 2));
  kp.resid = static_cast<const __nv_bfloat16*>(g.resid);
  if (kp.resid && g.epi != kEpiF32) return cudaErrorInvalidValue;
  kp.slice_rows = g.slice_rows;
  kp.vt_col0 = g.vt_col0;
  kp.mn_major = g.mn_major;
  // No narrow or chained MN-major products; 3-D maps only with their operand MN-major.
  if (g.mn_major && (g.chain || BN == 64)) return cudaErrorInvalidValue;
  if (((g.mn_major & kMnA3d) && !(g.mn_major & kMnA)) || ((g.mn_major & kMnB3d) && !(g.mn_major & kMnB)))
    return cudaErrorInvalidValue;
  if (g.slice_rows && (g.epi != kEpiF32 || !g.chain || g.resid)) return cudaErrorInvalidValue;
  if (!kp.status) return cudaErrorInvalidSymbol;
  if (kp.tiles == 0) return cudaSuccess;
  if (pair) {
    // Outputs with TMA maps leave the pair kernels through TMA stores.
    // (with rank slices only when no warp's 32 rows straddle two slices)
    // TPMLP_TMA_STORE: bit 0 the fp32 outputs, bit 1 the GeLU'd bf16 H (default both).
    const int tma_bits = env_int("TPMLP_TMA_STORE", 3);
    const bool tma_out = g.map_out[0] != nullptr && g.slice_rows % 32 == 0 &&
                         ((g.epi == kEpiF32 && (tma_bits & 1)) || (g.epi == kEpiGeluBf16 && (tma_bits & 2)));
    const int epi = !tma_out ? g.epi : g.epi == kEpiF32 ? kEpiF32Tma : kEpiGeluTma;
    return launch_pair(kp, epi, s);
  }
  if (BN == 64) return launch_single_epi<64>(kp, g.epi, s);
  return BN == 256 ? launch_single_epi<256>(kp, g.epi, s) : launch_single_epi<128>(kp, g.epi, s);
}

int num_sms() {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (!n) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n = v > 0 ? v : 1;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace tpmlp
