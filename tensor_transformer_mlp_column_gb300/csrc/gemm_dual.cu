// gemm_dual.cu — the backward's first step in one tcgen05 kernel: for every
// shard i and every 256 x 256 tile of [T, F/n], a CTA pair (cluster of two)
// recomputes the pre-activation P_i = X A_i and computes dH_i = dY B_i^T, both
// in tensor memory, and its epilogue writes H_i = GeLU(P_i) and
// dP_i = dH_i * GeLU'(P_i) (bf16, row-major). P never reaches global memory.
// This is the MLP backward of the tensor-parallel split (duoan.github.io
// "Tensor Parallelism in Megatron-LM" §3, the f/g operators: dY reaches every
// shard unchanged), with gelu' of the GPT-2 tanh form (scratchllm.com
// "Tensor-Parallel MLP (Megatron)", "GeLU").
//
// Tensor memory holds the two accumulators of one tile (P in columns 0..255,
// dH in 256..511), so the tile's two products run one after the other and the
// epilogue works in two phases that overlap the other product:
//   MMA  : P_t            | dH_t             | P_{t+1}          | dH_{t+1} ...
//   epi  :                | phase 1 of t     | phase 2 of t     | phase 1 of t+1 ...
// Phase 1 reads P, writes H and keeps GeLU'(P) as fp16 in registers, then
// releases the P accumulator; phase 2 reads dH, multiplies by the kept
// GeLU'(P), writes dP and releases the dH accumulator. GeLU' lies in
// (-0.17, 1.13), where fp16 keeps 11 significant bits, four times finer than
// the bf16 rounding of dP that follows.
//
// Roles (320 threads per CTA, one CTA per SM):
//   every CTA, warp 0 lane 0 : TMA producer; for each tile the K blocks of
//                              (X, A_i^T) and then of (dY, B_i), two 64-deep
//                              blocks per stage: its own 128 rows of X / dY
//                              and its 128 of the 256 rows of A_i^T / B_i,
//                              counted on the even CTA's barrier
//   even CTA, warp 1 lane 0  : MMA issuer (M = 256, N = 256, K = 16)
//   every CTA, warps 2..9    : epilogue of the CTA's own 128 rows, each warp
//                              32 rows x 128 columns
// Every wait is bounded; on a timeout the CTA raises the abort flag of its
// peer, all roles leave their loops, copies and MMAs in flight are drained and
// both CTAs free their tensor memory.
#include <cuda_fp16.h>

#include <atomic>
#include <cstring>
#include <type_traits>

#include "gemm_common.cuh"

namespace tpmlp {

namespace {

constexpr int kDualStages = 3;                       // stages of kDualKsub 64-deep K blocks
constexpr int kDualKsub = 2;
constexpr uint32_t kDualSub = 128 * BK * 2;          // one operand's 128 rows x 64 K (16 KB)
constexpr uint32_t kDualA = kDualKsub * kDualSub;    // a stage's M x K part
constexpr uint32_t kDualStageBytes = 2 * kDualA;     // M x K rows + this CTA's N x K rows
constexpr uint32_t kDualTmemCols = 512;              // P (0..255) and dH (256..511)
constexpr int kDualEpiWarps = 8;                     // two per TMEM lane quarter, one per 128-column half
constexpr int kDualThreads = 64 + 32 * kDualEpiWarps;
constexpr size_t kDualSmem = 1024 + size_t(kDualStages) * kDualStageBytes + 256;

struct DualParams {
  CUtensorMap map_x;                   // X  [T][D], 64 x 128 boxes
  CUtensorMap map_dy;                  // dY [T][D], 64 x 128 boxes
  CUtensorMap map_at[kMaxGroups];      // A_i^T [Fs][D], 64 x 128 boxes
  CUtensorMap map_b[kMaxGroups];       // B_i   [Fs][D], 64 x 128 boxes
  void* h[kMaxGroups];                 // H_i  bf16 [T][ldo]
  void* dp[kMaxGroups];                // dP_i bf16 [T][ldo]
  int64_t ldo;
  int M, N;
  TileGrid grid;
  int k_blocks, tiles;
  uint64_t wait_ns;
  int* status;
  int load_hint;
  int inject;  // test hook: > 0 withholds that stage fill (1-based) in every CTA
};

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kDualThreads, 1) tc_dual_bwd_kernel(const __grid_constant__ DualParams p) {
  constexpr int BN = 256;
  constexpr uint32_t kCtas = 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                                       // stages: M x K operand (X or dY)
  uint8_t* sB = smem + kDualStages * kDualA;                // stages: N x K operand (A_i^T or B_i)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kDualStages * kDualStageBytes);
  uint64_t* empty = full + kDualStages;
  uint64_t* acc_full = empty + kDualStages;  // [0] P complete, [1] dH complete
  uint64_t* acc_empty = acc_full + 2;        // [0] P read, [1] dH read (even CTA: 8 epilogue warps)
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t pos = rank & 1u;
  const uint32_t lead = 0;
  const int cluster = static_cast<int>(cluster_id_x());
  const int nclusters = static_cast<int>(cluster_count_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDualStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full + b, 1);
      mbar_init(acc_empty + b, 2 * kDualEpiWarps);  // even CTA: every epilogue warp of the pair
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.map_x);
    tma_prefetch_desc(&p.map_dy);
    for (int g = 0; g < p.grid.groups; ++g) {
      tma_prefetch_desc(&p.map_at[g]);
      tma_prefetch_desc(&p.map_b[g]);
    }
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, kDualTmemCols);
  tc_fence_before_sync();
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();
  const WaitGuard guard{abort_flag, p.wait_ns, p.status};
  const uint32_t abort_addr = smem_addr(const_cast<int*>(abort_flag));
  auto raise_abort_in_cluster = [&]() {
    for (uint32_t r = 0; r < kCtas; ++r)
      if (r != rank) st_cluster_u32(map_to_cta(abort_addr, r), 1u);
  };
  bool aborted = false;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (every CTA)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, parity_bits = 0;
      int fill = 0;
      const uint64_t pol_a = l2_policy(p.load_hint & 3), pol_b = l2_policy((p.load_hint >> 2) & 3);
      for (int tile = cluster; !aborted && tile < p.tiles; tile += nclusters) {
        int g, mb, nb;
        decode_tile(p.grid, tile, g, mb, nb);
        if (!tile_ok(p.grid, p.status, g, mb, nb)) continue;
        const int m0 = mb * 256 + static_cast<int>(pos) * 128;
        const int n0 = nb * BN + static_cast<int>(pos) * 128;
        for (int prod = 0; !aborted && prod < 2; ++prod) {
          const CUtensorMap* ma = prod == 0 ? &p.map_x : &p.map_dy;
          const CUtensorMap* mbmap = prod == 0 ? &p.map_at[g] : &p.map_b[g];
          for (int kb = 0; kb < p.k_blocks; kb += kDualKsub) {
            if (!wait_bounded(empty + stage, phase ^ 1u, guard, kSiteProducer)) {
              aborted = true;
              break;
            }
            const uint32_t full_lead = map_to_cta(smem_addr(full + stage), lead);
            const int nsub = p.k_blocks - kb < kDualKsub ? p.k_blocks - kb : kDualKsub;
            if (++fill != p.inject) {
              if (pos == 0) {
                mbar_arrive_expect_tx(full + stage, 2 * 2 * nsub * kDualSub);  // both CTAs' two operands
                armed |= 1u << stage;
                parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
              }
              for (int u = 0; u < nsub; ++u) {
                tma_load_2d_pair_hint(sA + stage * kDualA + u * kDualSub, ma, (kb + u) * BK, m0, full_lead, pol_a);
                tma_load_2d_pair_hint(sB + stage * kDualA + u * kDualSub, mbmap, (kb + u) * BK, n0, full_lead,
                                      pol_b);
              }
            }
            if (++stage == kDualStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (aborted) {
        raise_abort_in_cluster();
        if (pos == 0) {
          for (int s = 0; s < kDualStages; ++s)
            if (armed >> s & 1u) wait_drain(full + s, (parity_bits >> s) & 1u, p.wait_ns);
        } else {
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 200000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && pos == 0) {
      // ---------------- MMA issuer (even CTA of each pair)
      constexpr uint32_t IDESC = idesc_bf16_f32(256, BN);
      constexpr uint16_t kPairMask = 0x3;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;  // flips once per tile
      for (int tile = cluster; !aborted && tile < p.tiles; tile += nclusters) {
        if constexpr (kDebugBuild) {
          int g, mb, nb;
          decode_tile(p.grid, tile, g, mb, nb);
          if (!tile_ok(p.grid, p.status, g, mb, nb)) continue;
        }
        for (int prod = 0; !aborted && prod < 2; ++prod) {
          if (!wait_bounded(acc_empty + prod, acc_phase ^ 1u, guard, kSiteMmaAcc)) {
            aborted = true;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(prod * BN);
          for (int kb = 0; kb < p.k_blocks; kb += kDualKsub) {
            if (!wait_bounded(full + stage, phase, guard, kSiteMmaFull)) {
              aborted = true;
              break;
            }
            tc_fence_after_sync();
            const int nsub = p.k_blocks - kb < kDualKsub ? p.k_blocks - kb : kDualKsub;
            for (int u = 0; u < nsub; ++u) {
              const uint32_t a0 = smem_addr(sA + stage * kDualA + u * kDualSub);
              const uint32_t b0 = smem_addr(sB + stage * kDualA + u * kDualSub);
#pragma unroll
              for (int k = 0; k < BK / 16; ++k)
                tc_mma_bf16_pair(d_tmem, smem_desc_sw128(a0 + 32u * k), smem_desc_sw128(b0 + 32u * k), IDESC,
                                 (kb | u | k) != 0 ? 1u : 0u);
            }
            tc_commit_pair_multicast(empty + stage, kPairMask);
            if (++stage == kDualStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (aborted) break;
          tc_commit_pair_multicast(acc_full + prod, kPairMask);
        }
        acc_phase ^= 1u;
      }
      if (aborted) {
        raise_abort_in_cluster();
        tc_commit_pair_multicast(drain, static_cast<uint16_t>(1u << rank));
        wait_drain(drain, 0, p.wait_ns);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..9 of every CTA)
    // Warp w reads TMEM lane quarter w % 4 (rows 32 (w % 4) .. +31 of the CTA's
    // 128) and the 128-column half (w - 2) / 4 of both accumulators. Between
    // the two phases of a tile it keeps GeLU'(P) of its 32 x 128 block in
    // registers, as fp16 pairs (64 per thread).
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t acc_empty_lead = map_to_cta(smem_addr(acc_empty), lead);
    uint32_t acc_phase = 0;
    uint32_t gp[64];
    for (int tile = cluster; tile < p.tiles; tile += nclusters) {
      int g, mb, nb;
      decode_tile(p.grid, tile, g, mb, nb);
      if (!tile_ok(p.grid, p.status, g, mb, nb)) continue;
      const int64_t m = int64_t(mb) * 256 + int64_t(pos) * 128 + quarter * 32 + lane;
      const bool row_ok = m < p.M;
      const int c0 = half * 128;  // first column of this warp's half of the tile
      const uint32_t t_lanes = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(c0);
      __nv_bfloat16* hrow = static_cast<__nv_bfloat16*>(p.h[g]) + m * p.ldo + nb * BN + c0;
      __nv_bfloat16* dprow = static_cast<__nv_bfloat16*>(p.dp[g]) + m * p.ldo + nb * BN + c0;
      const int ncols = p.N - (nb * BN + c0);  // columns of this half inside the output (may be <= 0)
      // One phase: prod 0 reads P (writes H, keeps GeLU'(P)), prod 1 reads dH
      // (writes dP). Returns false if the accumulator's wait gave up.
      auto run_phase = [&](auto prod_c) -> bool {
        constexpr int prod = decltype(prod_c)::value;
        const bool ok = wait_bounded(acc_full + prod, acc_phase, guard, kSiteEpilogue);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) raise_abort_in_cluster();
          return false;
        }
        tc_fence_after_sync();
        const uint32_t t_acc = t_lanes + static_cast<uint32_t>(prod * BN);
        uint32_t r0[32];
        auto chunk = [&](int j, uint32_t (&v)[32]) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int col = 32 * j + 8 * q;
            float o[8];
            if constexpr (prod == 0) {
#pragma unroll
              for (int e = 0; e < 8; e += 2) {
                float d0, d1;
                gelu_and_grad_fast(__uint_as_float(v[8 * q + e]), o[e], d0);
                gelu_and_grad_fast(__uint_as_float(v[8 * q + e + 1]), o[e + 1], d1);
                gp[(col + e) >> 1] = pack_half2(d0, d1);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 8; e += 2) {
                const float2 gd = __half22float2(*reinterpret_cast<const __half2*>(&gp[(col + e) >> 1]));
                o[e] = __uint_as_float(v[8 * q + e]) * gd.x;
                o[e + 1] = __uint_as_float(v[8 * q + e + 1]) * gd.y;
              }
            }
            if (row_ok && col + 8 <= ncols)
              store16((prod == 0 ? hrow : dprow) + col,
                      make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                                 pack_bf16x2(o[6], o[7])),
                      false);
          }
        };
        // Four chunks of 32 columns (the other epilogue warps of the SM
        // sub-partition hide each load's latency).
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          __syncwarp();
          tmem_ld_32cols_issue(t_acc + static_cast<uint32_t>(32 * j), r0);
          tmem_ld_wait(r0);
          if (j == 3) {
            // Every column of this accumulator is in registers: hand it back.
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty_lead + 8u * static_cast<uint32_t>(prod));
          }
          chunk(j, r0);
        }
        return true;
      };
      if (!run_phase(std::integral_constant<int, 0>{})) break;
      if (!run_phase(std::integral_constant<int, 1>{})) break;
      acc_phase ^= 1u;
    }
  }

  tc_fence_before_sync();
  __syncwarp();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kDualTmemCols);
  }
}

}  // namespace

cudaError_t launch_dual_bwd(const DualBwd& d, uint64_t wait_ns, cudaStream_t s) {
  if (d.groups < 1 || d.groups > kMaxGroups || d.M < 0 || d.N < 8 || d.N % 8 != 0 || d.K < 1)
    return cudaErrorInvalidValue;
  DualParams p;
  memset(&p, 0, sizeof(p));
  p.map_x = *d.map_x;
  p.map_dy = *d.map_dy;
  for (int i = 0; i < d.groups; ++i) {
    p.map_at[i] = *d.map_at[i];
    p.map_b[i] = *d.map_b[i];
    p.h[i] = d.h[i];
    p.dp[i] = d.dp[i];
  }
  p.ldo = d.ldo;
  p.M = d.M;
  p.N = d.N;
  const int m_blocks = (d.M + 255) / 256, n_blocks = (d.N + 255) / 256;
  p.grid = TileGrid{0, kSharedA, d.groups, m_blocks, n_blocks, d.group_m};
  p.k_blocks = (d.K + BK - 1) / BK;
  p.tiles = m_blocks * n_blocks * d.groups;
  p.wait_ns = wait_ns;
  p.status = device_status_word();
  p.load_hint = d.load_hint;
  p.inject = d.inject;
  if (!p.status) return cudaErrorInvalidSymbol;
  if (p.tiles == 0) return cudaSuccess;

  auto kern = tc_dual_bwd_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kDualSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kDualThreads, 1, 1);
  cfg.dynamicSmemBytes = kDualSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  static std::atomic<int> max_clusters[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  int cached = max_clusters[dev].load(std::memory_order_relaxed);
  if (!cached) {
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    int n = 0;
    cfg.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    cfg.numAttrs = 2;
    if (e != cudaSuccess) return e;
    cached = n > 0 ? n : 1;
    max_clusters[dev].store(cached, std::memory_order_relaxed);
  }
  const int clusters = p.tiles < cached ? p.tiles : cached;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace tpmlp
