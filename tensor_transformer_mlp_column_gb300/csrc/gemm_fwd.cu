// gemm_fwd.cu — the bf16 forward's two products in one persistent launch of
// CTA pairs, for forwards of a few to a few tens of rounds of tiles whose
// weights stay in L2 (scratchllm.com "Tensor-Parallel MLP (Megatron)", "The
// split": H_i = GeLU(X A_i), Y_i = H_i B_i, summed in shard order).
//
// The tile list holds every tile of the first product (256 x 256 tiles of
// each shard's H_i = GeLU(X A_i), in bands of 256 token rows: all shards'
// column blocks of a band before the next band), then every tile of the
// second (the shard-ordered sum Y = sum_i H_i B_i, or the partials Y_i = H_i
// B_i, also band by band; a sum with fewer tiles than half the pairs in
// 256 x 128 tiles). Each CTA pair walks the list from its own index
// in steps of the pair count, so a pair whose first-product tiles are done
// starts on second-product tiles while other pairs finish the first product:
// the idle SMs of one product's last round work on the other.
//
// A second-product tile of band b reads H rows of band b, written by the
// epilogues of that band's first-product tiles on other SMs. Each epilogue
// warp, once its TMA stores of a first-product tile have completed, fences
// them to GPU scope and adds one to the band's counter in global memory; the
// producer of a second-product tile waits (bounded) until the counter shows
// every warp of every tile of the band, then orders its coming TMA reads
// after that observation with a proxy fence. A pair's tiles come in increasing list
// order, so all of its first-product tiles precede its second-product ones,
// and the grid never exceeds the clusters that can be resident at once:
// every counter a pair waits on is completed by pairs that never wait.
//
// Roles per CTA: warp 0 lane 0 the TMA producer, the even CTA's warp 1 lane 0
// the MMA issuer (M = 256, N = 256, K = 16), warps 2..9 the epilogue (GeLU ->
// bf16 H for the first product, fp32 for the second, both through
// shared-memory staging and TMA stores): two warps per TMEM lane quarter, one
// for each half of the 256 accumulator columns, so that the short tiles'
// epilogues (K = 768..1024 is only 12..16 K blocks of MMAs) keep up with the
// tensor cores. Every wait is bounded.
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "gemm_common.cuh"

namespace tpmlp {

namespace {

constexpr uint32_t kFwdSub = 128 * BK * 2;               // 128 rows x 64 K of one operand (16 KB)
constexpr int kFwdKsub = 2;                              // K blocks per stage
constexpr int kFwdStages = 3;
constexpr uint32_t kFwdHalf = kFwdKsub * kFwdSub;        // a stage's M x K (or N x K) part
constexpr uint32_t kFwdStageBytes = 2 * kFwdHalf;
constexpr int kFwdEpiWarps = 8;                          // two per TMEM lane quarter
constexpr int kFwdThreads = 64 + 32 * kFwdEpiWarps;      // producer warp, MMA warp, epilogue warps
constexpr uint32_t kFwdOutBlock = 32 * 128;              // 32 rows of 128 bytes: 32 fp32 or 64 bf16 columns
constexpr uint32_t kFwdStaging = kFwdEpiWarps * kFwdOutBlock;  // one per epilogue warp
constexpr uint32_t kFwdTmemCols = 512;                   // two accumulators of 256 columns
constexpr size_t kFwdSmem = 1024 + size_t(kFwdStages) * kFwdStageBytes + kFwdStaging + 256;

struct FwdParams {
  CUtensorMap map_x;                // X [T][D], 64 x 128 boxes
  CUtensorMap map_at[kMaxGroups];   // A_i^T [Fs][D], 64 x 128 boxes
  CUtensorMap map_h[kMaxGroups];    // H_i [T][Fs], 64 x 128 boxes (the second product's M x K operand)
  CUtensorMap map_bt[kMaxGroups];   // B_i^T [D][Fs], 64 x 128 boxes
  CUtensorMap map_bt64[kMaxGroups]; // the same in 64 x 64 boxes (second-product tiles 128 wide)
  CUtensorMap map_out[kMaxGroups];  // fp32 outputs in 32 x 32 boxes: Y ([0], chain) or Y_i
  CUtensorMap map_hs[kMaxGroups];   // H_i as the first product's output, bf16 in 64 x 32 boxes
  void* h[kMaxGroups];              // H_i, bf16 [T][Fs]
  int M, N1, N2;                    // T, F/n, D
  int groups, chain;
  int m_blocks, n_blocks1, n_blocks2, k_blocks1, k_blocks2;
  int bn2;            // width of the second product's tiles: 256, or 128 for a short shard-ordered sum
  int tiles1, tiles;
  int band_arrivals;  // epilogue-warp arrivals that complete a band of H
  int* band_done;     // [m_blocks] counters, zero at launch
  uint64_t wait_ns;
  int* status;
  int load_hint;
};

struct FwdTile {
  int second;  // 0: H_i = GeLU(X A_i); 1: the second product
  int g, mb, nb;
};

__device__ __forceinline__ FwdTile decode_fwd(const FwdParams& p, int t) {
  FwdTile f;
  if (t < p.tiles1) {
    const int cols = p.groups * p.n_blocks1;
    const int c = t % cols;
    f.second = 0;
    f.mb = t / cols;
    f.g = c / p.n_blocks1;
    f.nb = c % p.n_blocks1;
    return f;
  }
  t -= p.tiles1;
  f.second = 1;
  if (p.chain) {
    f.g = 0;
    f.mb = t / p.n_blocks2;
    f.nb = t % p.n_blocks2;
    return f;
  }
  const int cols = p.groups * p.n_blocks2;
  const int c = t % cols;
  f.mb = t / cols;
  f.g = c / p.n_blocks2;
  f.nb = c % p.n_blocks2;
  return f;
}

// Debug build: the tile lies inside its product's grid.
__device__ __forceinline__ bool fwd_tile_ok(const FwdParams& p, const FwdTile& f) {
  return TPMLP_DCHECK(f.mb >= 0 && f.mb < p.m_blocks && f.g >= 0 && f.g < p.groups && f.nb >= 0 &&
                          f.nb < (f.second ? p.n_blocks2 : p.n_blocks1),
                      p.status, kChkTile);
}

// Waits until *ctr >= target (acquire, GPU scope), polling with short sleeps;
// gives up like wait_bounded after the time limit or on the CTA's abort flag.
__device__ __forceinline__ bool wait_counter(const int* ctr, int target, const WaitGuard& g, int site) {
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if (*g.abort_flag) return false;
    if (global_timer_ns() - t0 > g.limit_ns) {
      *g.abort_flag = 1;
      atomicCAS(g.status, 0, site);
      return false;
    }
    __nanosleep(200);
  }
}

static_assert(sizeof(FwdParams) <= 32764, "kernel parameters above the 32764-byte limit");

__global__ void __launch_bounds__(kFwdThreads, 1) tc_fwd_persistent_kernel(const __grid_constant__ FwdParams p) {
  constexpr int BN = 256;
  constexpr uint32_t kCtas = 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kFwdStages * kFwdHalf;
  uint8_t* s_out = smem + kFwdStages * kFwdStageBytes;  // 1024-aligned TMA-store staging
  uint64_t* full = reinterpret_cast<uint64_t*>(s_out + kFwdStaging);
  uint64_t* empty = full + kFwdStages;
  uint64_t* acc_full = empty + kFwdStages;
  uint64_t* acc_empty = acc_full + 2;
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
    for (int s = 0; s < kFwdStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full + b, 1);
      mbar_init(acc_empty + b, 2 * kFwdEpiWarps);  // every epilogue warp of the pair
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.map_x);
    for (int g = 0; g < p.groups; ++g) {
      tma_prefetch_desc(&p.map_at[g]);
      tma_prefetch_desc(&p.map_h[g]);
      tma_prefetch_desc(&p.map_bt[g]);
    }
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, kFwdTmemCols);
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
  // K blocks of a tile: the first product contracts over D, the second over
  // F/n (per shard, all shards in order when chained).
  auto k_blocks_of = [&](const FwdTile& f) {
    return f.second ? (p.chain ? p.groups * p.k_blocks2 : p.k_blocks2) : p.k_blocks1;
  };
  bool aborted = false;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (every CTA)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, parity_bits = 0;
      const uint64_t pol_a = l2_policy(p.load_hint & 3), pol_b = l2_policy((p.load_hint >> 2) & 3);
      for (int tile = cluster; !aborted && tile < p.tiles; tile += nclusters) {
        const FwdTile f = decode_fwd(p, tile);
        if (!fwd_tile_ok(p, f)) continue;
        if (f.second) {
          // The band's rows of every H_i must be written: wait for all of the
          // band's first-product epilogue warps, then order the TMA reads of H
          // (async proxy) after that observation.
          if (!wait_counter(p.band_done + f.mb, p.band_arrivals, guard, kSiteBand)) {
            aborted = true;
            break;
          }
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        const int tbn = f.second ? p.bn2 : BN;  // the tile's width; each CTA loads half of its N x K rows
        const bool narrow = tbn != BN;
        const int m0 = f.mb * 256 + static_cast<int>(pos) * 128;
        const int n0 = f.nb * tbn + static_cast<int>(pos) * (tbn / 2);
        const int kb_tile = k_blocks_of(f);
        const int kb_group = f.second ? p.k_blocks2 : p.k_blocks1;
        int gg = f.g, kk = 0;
        for (int kb = 0; kb < kb_tile; kb += kFwdKsub) {
          if (!wait_bounded(empty + stage, phase ^ 1u, guard, kSiteProducer)) {
            aborted = true;
            break;
          }
          const uint32_t full_lead = map_to_cta(smem_addr(full + stage), lead);
          const int nsub = kb_tile - kb < kFwdKsub ? kb_tile - kb : kFwdKsub;
          if (!TPMLP_DCHECK((kk * BK) % 8 == 0 && m0 % 64 == 0 && n0 % 64 == 0, p.status, kChkTmaX)) {
            aborted = true;
            break;
          }
          if (pos == 0) {
            mbar_arrive_expect_tx(full + stage, 2 * nsub * (kFwdSub + (narrow ? kFwdSub / 2 : kFwdSub)));  // both CTAs' A and B
            armed |= 1u << stage;
            parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
          }
          for (int u = 0; u < nsub; ++u) {
            const CUtensorMap* ma = f.second ? &p.map_h[gg] : &p.map_x;
            const CUtensorMap* mbm = !f.second ? &p.map_at[gg] : narrow ? &p.map_bt64[gg] : &p.map_bt[gg];
            tma_load_2d_pair_hint(sA + stage * kFwdHalf + u * kFwdSub, ma, kk * BK, m0, full_lead, pol_a);
            tma_load_2d_pair_hint(sB + stage * kFwdHalf + u * kFwdSub, mbm, kk * BK, n0, full_lead, pol_b);
            if (++kk == kb_group) {
              kk = 0;
              ++gg;
            }
          }
          if (++stage == kFwdStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (aborted) {
        raise_abort_in_cluster();
        if (pos == 0) {
          for (int s = 0; s < kFwdStages; ++s)
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
      constexpr uint32_t IDESC_NARROW = idesc_bf16_f32(256, BN / 2);
      constexpr uint16_t kPairMask = 0x3;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int tile = cluster; !aborted && tile < p.tiles; tile += nclusters) {
        const FwdTile f = decode_fwd(p, tile);
        if (!fwd_tile_ok(p, f)) continue;
        if (!wait_bounded(acc_empty + acc, acc_phase ^ 1u, guard, kSiteMmaAcc)) {
          aborted = true;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        const int kb_tile = k_blocks_of(f);
        const uint32_t idesc = (f.second && p.bn2 != BN) ? IDESC_NARROW : IDESC;
        for (int kb = 0; kb < kb_tile; kb += kFwdKsub) {
          if (!wait_bounded(full + stage, phase, guard, kSiteMmaFull)) {
            aborted = true;
            break;
          }
          tc_fence_after_sync();
          const int nsub = kb_tile - kb < kFwdKsub ? kb_tile - kb : kFwdKsub;
          for (int u = 0; u < nsub; ++u) {
            const uint32_t a0 = smem_addr(sA + stage * kFwdHalf + u * kFwdSub);
            const uint32_t b0 = smem_addr(sB + stage * kFwdHalf + u * kFwdSub);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              tc_mma_bf16_pair(d_tmem, smem_desc_sw128(a0 + 32u * k), smem_desc_sw128(b0 + 32u * k), idesc,
                               (kb | u | k) != 0 ? 1u : 0u);
          }
          tc_commit_pair_multicast(empty + stage, kPairMask);
          if (++stage == kFwdStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (aborted) break;
        tc_commit_pair_multicast(acc_full + acc, kPairMask);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (aborted) {
        raise_abort_in_cluster();
        tc_commit_pair_multicast(drain, static_cast<uint16_t>(1u << rank));
        wait_drain(drain, 0, p.wait_ns);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..9 of every CTA)
    const int quarter = warp & 3;      // TMEM lanes (rows) quarter*32 .. +31
    const int half_col = (warp - 2) >> 2;  // which half of the tile's accumulator columns this warp takes
    uint8_t* const buf = s_out + (warp - 2) * kFwdOutBlock;
    const uint32_t acc_empty_lead = map_to_cta(smem_addr(acc_empty), lead);
    int acc = 0;
    uint32_t acc_phase = 0;
    int blocks_out = 0;  // staging blocks this warp has handed to TMA so far
    for (int tile = cluster; tile < p.tiles; tile += nclusters) {
      const FwdTile f = decode_fwd(p, tile);
      if (!fwd_tile_ok(p, f)) continue;
      const bool ok = wait_bounded(acc_full + acc, acc_phase, guard, kSiteEpilogue);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) raise_abort_in_cluster();
        break;
      }
      tc_fence_after_sync();
      const int64_t m_warp = int64_t(f.mb) * 256 + int64_t(pos) * 128 + quarter * 32;
      const int N = f.second ? p.N2 : p.N1;
      const int tbn = f.second ? p.bn2 : BN;
      const int col0 = half_col * (tbn / 2), col1 = col0 + tbn / 2;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
      auto finish = [&](int c, const uint32_t (&r)[32]) {
        const int n0 = f.nb * tbn + c;
        if (!f.second) {
          // H = GeLU(acc) in bf16, staged as the warp's 32 x 64 block (128-byte
          // rows, 128-byte swizzle: 16-byte unit u of row r at u ^ (r % 8)),
          // two 32-column chunks per block, then one TMA store of the block
          // (clipped to T x F/n): whole lines instead of each lane writing its
          // own row.
          const int half = (c >> 5) & 1;
          const int nb0 = n0 - 32 * half;  // the block's first column (a multiple of 64)
          if (nb0 >= N || m_warp >= p.M) return;  // warp-uniform, the same for both chunks of a block
          // (checked for both chunks, so that a failed check skips the whole block)
          if (!TPMLP_DCHECK(nb0 % 64 == 0 && m_warp % 32 == 0 && nb0 >= 0 && m_warp >= 0, p.status, kChkOutput))
            return;
          if (half == 0) {
            if (blocks_out >= 1 && lane == 0) bulk_wait_group_read<0>();  // the previous store has read the buffer
            __syncwarp();
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = gelu_bf16_fast(__uint_as_float(r[8 * j + e]));
            *reinterpret_cast<uint4*>(buf + lane * 128 + (((4 * half + j) ^ (lane & 7)) << 4)) =
                make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                           pack_bf16x2(x[6], x[7]));
          }
          if (half == 1) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&p.map_hs[f.g], buf, nb0, static_cast<int32_t>(m_warp));
              bulk_commit_group();
            }
            ++blocks_out;
          }
          return;
        }
        // fp32 through a TMA store of the warp's 32 x 32 block (128-byte swizzled staging).
        if (n0 >= N || m_warp >= p.M) return;  // warp-uniform
        if (!TPMLP_DCHECK(n0 % 32 == 0 && m_warp % 32 == 0, p.status, kChkOutput)) return;
        if (blocks_out >= 1 && lane == 0) bulk_wait_group_read<0>();  // the previous store has read the buffer
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
              make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&p.map_out[p.chain ? 0 : f.g], buf, n0, static_cast<int32_t>(m_warp));
          bulk_commit_group();
        }
        ++blocks_out;
      };
      uint32_t ra[32], rb[32];
      __syncwarp();
      tmem_ld_32cols_issue(t_row + static_cast<uint32_t>(col0), ra);
      tmem_ld_wait(ra);
#pragma unroll 1
      for (int c = col0; c < col1; c += 64) {
        __syncwarp();
        tmem_ld_32cols_issue(t_row + static_cast<uint32_t>(c + 32), rb);
        finish(c, ra);
        __syncwarp();
        tmem_ld_wait(rb);
        if (c + 64 == col1) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty_lead + 8u * static_cast<uint32_t>(acc));
        } else {
          __syncwarp();
          tmem_ld_32cols_issue(t_row + static_cast<uint32_t>(c + 64), ra);
        }
        finish(c + 32, rb);
        if (c + 64 < col1) {
          __syncwarp();
          tmem_ld_wait(ra);
        }
      }
      if (!f.second) {
        // This warp's rows of the band are written once its TMA stores have
        // completed: then make them visible at GPU scope (the async-proxy
        // writes ordered before the generic release) and count the warp in
        // the band.
        if (lane == 0) {
          bulk_wait_group_all();
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __threadfence();
          atomicAdd(p.band_done + f.mb, 1);
        }
        __syncwarp();
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_group_all();  // every store has left shared memory and landed
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncwarp();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kFwdTmemCols);
  }
}

// Zeroes the band counters of the next launch. Launched with programmatic
// dependent launch like the kernels around it: it waits for the previous
// kernel of the stream before writing, and the forward kernel's own wait
// covers its writes.
__global__ void zero_counters_kernel(int* ctr, int n) {
  pdl_wait();
  pdl_launch_dependents();
  for (int i = threadIdx.x; i < n; i += blockDim.x) ctr[i] = 0;
}

}  // namespace

int fwd_second_width(int64_t M, int64_t N2, int chain) {
  static const int narrow = [] {
    const char* e = getenv("TPMLP_FWD_NARROW2");
    return (e && *e) ? atoi(e) : 1;
  }();
  if (!chain || !narrow) return 256;
  // Half-width tiles load 1.5 times the bytes per MMA of full ones: they pay
  // only while the sum's tiles leave most pairs idle (the narrow tiles still
  // fit one round), not when every SM is loading from L2 at once.
  const int64_t tiles = ((M + 255) / 256) * ((N2 + 255) / 256);
  const int pairs = fwd_persistent_clusters();
  return 2 * tiles <= pairs ? 128 : 256;
}

int fwd_persistent_clusters() {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaFuncSetAttribute(tc_fwd_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kFwdSmem)) != cudaSuccess)
      return 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    cfg.blockDim = dim3(kFwdThreads, 1, 1);
    cfg.dynamicSmemBytes = kFwdSmem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int v = 0;
    if (cudaOccupancyMaxActiveClusters(&v, tc_fwd_persistent_kernel, &cfg) != cudaSuccess || v < 1) return 0;
    n = v;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

cudaError_t launch_fwd_persistent(const FwdPersistent& f, uint64_t wait_ns, cudaStream_t s) {
  if (f.groups < 1 || f.groups > kMaxGroups || f.M < 1 || f.N1 < 8 || f.N2 < 8 || f.K1 < 1 || !f.band_done)
    return cudaErrorInvalidValue;
  FwdParams p;
  memset(&p, 0, sizeof(p));
  p.map_x = *f.map_x;
  for (int i = 0; i < f.groups; ++i) {
    p.map_at[i] = *f.map_at[i];
    p.map_h[i] = *f.map_h[i];
    p.map_bt[i] = *f.map_bt[i];
    p.map_bt64[i] = *f.map_bt64[i];
    p.h[i] = f.h[i];
  }
  for (int i = 0; i < (f.chain ? 1 : f.groups); ++i) p.map_out[i] = *f.map_out[i];
  for (int i = 0; i < f.groups; ++i)
    if (!make_output_map_bf16(&p.map_hs[i], f.h[i], f.M, f.N1, f.N1)) return cudaErrorInvalidValue;
  p.M = f.M;
  p.N1 = f.N1;
  p.N2 = f.N2;
  p.groups = f.groups;
  p.chain = f.chain;
  p.m_blocks = (f.M + 255) / 256;
  p.n_blocks1 = (f.N1 + 255) / 256;
  p.bn2 = fwd_second_width(f.M, f.N2, f.chain);
  p.n_blocks2 = (f.N2 + p.bn2 - 1) / p.bn2;
  p.k_blocks1 = (f.K1 + BK - 1) / BK;
  p.k_blocks2 = (f.N1 + BK - 1) / BK;
  p.tiles1 = p.m_blocks * p.n_blocks1 * f.groups;
  p.tiles = p.tiles1 + p.m_blocks * p.n_blocks2 * (f.chain ? 1 : f.groups);
  p.band_arrivals = p.n_blocks1 * f.groups * 2 * kFwdEpiWarps + f.band_extra;  // every epilogue warp of the pair
  p.band_done = f.band_done;
  p.wait_ns = wait_ns;
  p.status = device_status_word();
  p.load_hint = 1 | (1 << 2);
  if (!p.status) return cudaErrorInvalidSymbol;
  const int clusters_max = fwd_persistent_clusters();
  if (clusters_max < 1) return cudaErrorInvalidConfiguration;
  cudaError_t e = launch_pdl(zero_counters_kernel, dim3(1), dim3(128), 0, s, f.band_done, p.m_blocks);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  // Never more pairs than can be resident at once: a pair may wait for bands
  // that other pairs write.
  const int clusters = p.tiles < clusters_max ? p.tiles : clusters_max;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(kFwdThreads, 1, 1);
  cfg.dynamicSmemBytes = kFwdSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, tc_fwd_persistent_kernel, p);
}

}  // namespace tpmlp
