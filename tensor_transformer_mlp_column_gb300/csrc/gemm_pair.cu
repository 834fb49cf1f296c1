// gemm_pair.cu — tcgen05 cta_group::2 GEMM: a CTA pair (cluster of 2 CTAs on
// two SMs) computes one 256 x 256 tile.
//
// Per k-block each CTA brings in its 128 rows of the M x K operand and its
// 128 of the 256 rows of the N x K operand (the pair MMA reads both CTAs'
// shared memory); every CTA loads only into its own shared memory. An
// operand may be K-major (one 64 x 128 box) or MN-major (a row-major [K][M]
// tensor: two 64-wide chunks of 64 K rows), so products with a transposed
// operand read it in place.
//   every CTA, warp 0 lane 0 : TMA producer; the pair's bytes are counted on
//                              the full barrier of the pair's even CTA, which
//                              its producer arms with both CTAs' bytes
//   even CTA, warp 1 lane 0  : MMA issuer (M=256, N=256, K=16 per
//                              instruction) into one of two TMEM accumulators;
//                              commits free each stage in both CTAs and
//                              publish each accumulator in the pair
//   every CTA, warps 2..5    : epilogue of the CTA's own 128 rows; release the
//                              accumulator on the pair's even CTA
// Every wait is bounded; on a timeout the CTA raises the abort flag of the
// other CTA of its pair, all roles leave their loops, copies in flight and
// MMAs are drained, and both CTAs free their TMEM.
#include "gemm_common.cuh"

#include <atomic>

namespace tpmlp {

namespace {

// A stage holds KSUB = 2 consecutive 64-column K blocks (each a 128-row tile
// of 128-byte swizzled rows): three stages of 64 KB, half the barrier round
// trips per MMA of one-block stages; the TMA-store epilogue's 32 KB of output
// staging still fits beside them.
constexpr uint32_t kSubBytes = 128 * BK * 2;
template <int EPI>
constexpr int ksub_of() {
  return 2;
}
template <int EPI>
constexpr int stages_of() {
  return 3;
}

template <int STAGES_, int KSUB_>
struct PairCfg {
  static constexpr int STAGES = STAGES_;
  static constexpr int KSUB = KSUB_;
  static constexpr uint32_t A_BYTES = KSUB * kSubBytes;  // this CTA's 128 rows
  static constexpr uint32_t B_BYTES = KSUB * kSubBytes;  // this CTA's half of the 256 N rows
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TMEM_COLS = 512;  // two accumulators of 256 fp32 columns
  // TMA-store epilogues: two 4 KB staging blocks per epilogue warp (32 rows
  // of 128 bytes: 32 fp32 or 64 bf16 columns).
  static constexpr uint32_t OUT_BLOCK = 32 * 128;
  template <int EPI>
  static constexpr uint32_t staging() {
    return (EPI == kEpiF32Tma || EPI == kEpiGeluTma) ? 4 * 2 * OUT_BLOCK : 0;
  }
  template <int EPI>
  static constexpr size_t smem() {
    return 1024 + size_t(STAGES) * STAGE_BYTES + staging<EPI>() + 256;
  }
};

template <int EPI, int STAGES>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_pair_kernel(const __grid_constant__ KParams p) {
  using C = PairCfg<STAGES, ksub_of<EPI>()>;
  constexpr int BN = 256;
  constexpr uint32_t kCtas = 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  uint8_t* s_out = smem + C::STAGES * C::STAGE_BYTES;  // 1024-aligned staging of the TMA-store epilogues
  uint64_t* full = reinterpret_cast<uint64_t*>(s_out + C::template staging<EPI>());
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t pos = rank & 1u;   // position in the pair: 0 = even CTA, issues the pair's MMAs
  const uint32_t lead = 0;          // the pair's even CTA
  const int cluster = static_cast<int>(cluster_id_x());
  const int nclusters = static_cast<int>(cluster_count_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full + s, 1);                    // even CTA: its producer's arrive (+ the pair's bytes)
      mbar_init(empty + s, 1);                   // the pair's commit once its MMAs have read the stage
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full + b, 1);   // one commit per tile
      mbar_init(acc_empty + b, 8);  // even CTA: one arrival per epilogue warp of the pair
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int g = 0; g < p.groups; ++g) {
      tma_prefetch_desc(&p.map_a[g]);
      tma_prefetch_desc(&p.map_b[g]);
    }
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
  tc_fence_before_sync();
  cluster_sync_all();  // barriers of every CTA initialised, TMEM allocated
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // Set-up done: from here on global memory is read and written, so wait for
  // the previous kernel of the stream, and let the next one start its set-up.
  pdl_wait();
  pdl_launch_dependents();
  const WaitGuard guard{abort_flag, p.wait_ns, p.status};
  const uint32_t abort_addr = smem_addr(const_cast<int*>(abort_flag));
  auto raise_abort_in_cluster = [&]() {
    for (uint32_t r = 0; r < kCtas; ++r)
      if (r != rank) st_cluster_u32(map_to_cta(abort_addr, r), 1u);
  };
  const int kb_per_tile = p.chain ? p.groups * p.k_blocks : p.k_blocks;
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
        decode_tile(p, tile, g, mb, nb);
        if (!tile_ok(p, g, mb, nb)) continue;
        const int m0 = mb * 256 + static_cast<int>(pos) * 128;
        const int n0 = nb * BN + static_cast<int>(pos) * 128;
        int gg = g, kk = 0;  // group and K block of the next load (chain mode walks the groups in order)
        for (int kb = 0; kb < kb_per_tile; kb += C::KSUB) {
          if (!wait_bounded(empty + stage, phase ^ 1u, guard, kSiteProducer)) {
            aborted = true;
            break;
          }
          const uint32_t full_lead = map_to_cta(smem_addr(full + stage), lead);
          const int nsub = kb_per_tile - kb < C::KSUB ? kb_per_tile - kb : C::KSUB;  // K blocks in this stage
          ++fill;
          // Inner (x) coordinates of this stage's loads must be 16-byte aligned
          // (K-major: kk * BK; MN-major: m0, n0; 3-D maps: chunk starts).
          if (!TPMLP_DCHECK((kk * BK) % 8 == 0 && m0 % 64 == 0 && n0 % 64 == 0, p.status, kChkTmaX)) {
            aborted = true;
            break;
          }
          if (fill != p.inject) {
            if (pos == 0) {
              mbar_arrive_expect_tx(full + stage, 2 * 2 * nsub * kSubBytes);  // both CTAs' A and B
              armed |= 1u << stage;
              parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
            }
            for (int u = 0; u < nsub; ++u) {
              uint8_t* da = sA + stage * C::A_BYTES + u * kSubBytes;
              uint8_t* db = sB + stage * C::B_BYTES + u * kSubBytes;
              // MN-major operands ([K][M] tensors) arrive as two 64-wide chunks of
              // 64 K rows: one box of a 3-D map (chunk index z = m0 / 64) or two
              // boxes of a 2-D one.
              if (p.mn_major & kMnA3d) {
                tma_load_3d_pair_hint(da, &p.map_a[gg], 0, kk * BK, m0 / 64, full_lead, pol_a);
              } else if (p.mn_major & kMnA) {
                tma_load_2d_pair_hint(da, &p.map_a[gg], m0, kk * BK, full_lead, pol_a);
                tma_load_2d_pair_hint(da + kMnChunkBytes, &p.map_a[gg], m0 + 64, kk * BK, full_lead, pol_a);
              } else {
                tma_load_2d_pair_hint(da, &p.map_a[gg], kk * BK, m0, full_lead, pol_a);
              }
              if (p.mn_major & kMnB3d) {
                tma_load_3d_pair_hint(db, &p.map_b[gg], 0, kk * BK, n0 / 64, full_lead, pol_b);
              } else if (p.mn_major & kMnB) {
                tma_load_2d_pair_hint(db, &p.map_b[gg], n0, kk * BK, full_lead, pol_b);
                tma_load_2d_pair_hint(db + kMnChunkBytes, &p.map_b[gg], n0 + 64, kk * BK, full_lead, pol_b);
              } else {
                tma_load_2d_pair_hint(db, &p.map_b[gg], kk * BK, n0, full_lead, pol_b);
              }
              if (++kk == p.k_blocks) {
                kk = 0;
                ++gg;
              }
            }
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
      if (aborted) {
        raise_abort_in_cluster();
        if (pos == 0) {
          for (int s = 0; s < C::STAGES; ++s)
            if (armed >> s & 1u) wait_drain(full + s, (parity_bits >> s) & 1u, p.wait_ns);
        } else {
          // This CTA's copies are counted on the even CTA's barriers; give any
          // copy still in flight time to land before shared memory is released.
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 200000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && pos == 0) {
      // ---------------- MMA issuer (even CTA of each pair)
      const bool a_mn = (p.mn_major & kMnA) != 0, b_mn = (p.mn_major & kMnB) != 0;
      const uint32_t idesc = idesc_bf16_f32(256, BN, a_mn, b_mn);
      constexpr uint16_t kPairMask = 0x3;  // both CTAs: each holds half of every stage and of every accumulator
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int tile = cluster; !aborted && tile < p.tiles; tile += nclusters) {
        if constexpr (kDebugBuild) {
          int g, mb, nb;
          decode_tile(p, tile, g, mb, nb);
          if (!tile_ok(p, g, mb, nb)) continue;
        }
        if (!wait_bounded(acc_empty + acc, acc_phase ^ 1u, guard, kSiteMmaAcc)) {
          aborted = true;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < kb_per_tile; kb += C::KSUB) {
          if (!wait_bounded(full + stage, phase, guard, kSiteMmaFull)) {
            aborted = true;
            break;
          }
          tc_fence_after_sync();
          const int nsub = kb_per_tile - kb < C::KSUB ? kb_per_tile - kb : C::KSUB;
          for (int u = 0; u < nsub; ++u) {
            const uint32_t a0 = smem_addr(sA + stage * C::A_BYTES + u * kSubBytes);
            const uint32_t b0 = smem_addr(sB + stage * C::B_BYTES + u * kSubBytes);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              tc_mma_bf16_pair(d_tmem, operand_desc(a0, k, a_mn), operand_desc(b0, k, b_mn), idesc,
                               (kb | u | k) != 0 ? 1u : 0u);
            }
          }
          tc_commit_pair_multicast(empty + stage, kPairMask);  // frees the stage once these MMAs have read it
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (aborted) break;
        tc_commit_pair_multicast(acc_full + acc, kPairMask);  // accumulator complete in both CTAs of the pair
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
    // ---------------- epilogue (warps 2..5 of every CTA)
    const int quarter = warp & 3;  // rows quarter*32 .. +31 of this CTA's 128 (its TMEM lane quarter)
    const uint32_t acc_empty_lead = map_to_cta(smem_addr(acc_empty), lead);
    int acc = 0;
    uint32_t acc_phase = 0;
    int blocks_out = 0;  // TMA-store epilogues: staging blocks this warp has handed to TMA so far
    for (int tile = cluster; tile < p.tiles; tile += nclusters) {
      int g, mb, nb;
      decode_tile(p, tile, g, mb, nb);
      if (!tile_ok(p, g, mb, nb)) continue;
      bool ok = wait_bounded(acc_full + acc, acc_phase, guard, kSiteEpilogue);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) raise_abort_in_cluster();
        break;
      }
      tc_fence_after_sync();
      const int64_t m_warp = int64_t(mb) * 256 + int64_t(pos) * 128 + quarter * 32;  // row of lane 0
      const int64_t m = m_warp + lane;
      const bool row_ok = m < p.M;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
      // The 256 columns in chunks of 32, software-pipelined: the tcgen05.ld
      // of the next chunk (and its residual load) is in flight while the
      // current chunk is converted and stored.
      auto with_res = [&](int n0) {
        return (EPI == kEpiF32 || EPI == kEpiF32Tma) && p.resid != nullptr && row_ok && n0 < p.N;
      };
      auto issue = [&](int c, uint32_t (&r)[32], uint4 (&res)[4]) {
        const int n0 = nb * BN + c;
        if (with_res(n0)) load_residual(p, m, n0, res);
        __syncwarp();
        tmem_ld_32cols_issue(t_row + static_cast<uint32_t>(c), r);
      };
      auto finish = [&](int c, const uint32_t (&r)[32], const uint4 (&res)[4]) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
        const int n0 = nb * BN + c;
        if (with_res(n0)) add_residual(res, v);
        if constexpr (EPI == kEpiF32Tma) {
          // Stage the warp's 32 x 32 fp32 block in shared memory with the
          // 128-byte swizzle (16-byte chunk j of row r at slot j ^ (r % 8),
          // conflict-free for these row-per-lane writes), then one TMA store
          // writes it as whole 128-byte lines, clipped to M x N.
          if (n0 >= p.N || m_warp >= p.M) return;  // warp-uniform
          if (!TPMLP_DCHECK(n0 % 32 == 0 && m_warp % 32 == 0 && n0 >= 0 && m_warp >= 0, p.status, kChkOutput)) return;
          uint8_t* buf = s_out + (quarter * 2 + (blocks_out & 1)) * C::OUT_BLOCK;
          if (blocks_out >= 2 && lane == 0) bulk_wait_group_read<1>();  // this buffer's previous store has read it
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]), __float_as_uint(v[4 * j + 2]),
                           __float_as_uint(v[4 * j + 3]));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            // Rank slices (slice_rows % 32 == 0): the warp's 32 rows lie in one
            // slice, whose own map takes the row within the slice.
            const int map = p.slice_rows ? static_cast<int>(m_warp / p.slice_rows) : g;
            const int64_t row = p.slice_rows ? m_warp % p.slice_rows : m_warp;
            tma_store_2d(&p.map_out[map], buf, n0, static_cast<int32_t>(row));
            bulk_commit_group();
          }
          ++blocks_out;
        } else if constexpr (EPI == kEpiGeluTma) {
          // GeLU'd bf16: the warp's 32 x 64 block (128-byte rows, the same
          // swizzle) takes two 32-column chunks, then one TMA store writes it,
          // clipped to M x N.
          const int half = (c >> 5) & 1;
          const int nb0 = n0 - 32 * half;  // the block's first column, a multiple of 64
          if (nb0 >= p.N || m_warp >= p.M) return;  // warp-uniform, the same for both chunks of a block
          // (checked for both chunks, so that a failed check skips the whole block)
          if (!TPMLP_DCHECK(nb0 % 64 == 0 && m_warp % 32 == 0 && nb0 >= 0 && m_warp >= 0, p.status, kChkOutput))
            return;
          uint8_t* buf = s_out + (quarter * 2 + (blocks_out & 1)) * C::OUT_BLOCK;
          if (half == 0) {
            if (blocks_out >= 2 && lane == 0) bulk_wait_group_read<1>();  // this buffer's previous store has read it
            __syncwarp();
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(buf + lane * 128 + (((4 * half + j) ^ (lane & 7)) << 4)) =
                make_uint4(pack_bf16x2(gelu_bf16_fast(v[8 * j]), gelu_bf16_fast(v[8 * j + 1])),
                           pack_bf16x2(gelu_bf16_fast(v[8 * j + 2]), gelu_bf16_fast(v[8 * j + 3])),
                           pack_bf16x2(gelu_bf16_fast(v[8 * j + 4]), gelu_bf16_fast(v[8 * j + 5])),
                           pack_bf16x2(gelu_bf16_fast(v[8 * j + 6]), gelu_bf16_fast(v[8 * j + 7])));
          if (half == 1) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&p.map_out[g], buf, nb0, static_cast<int32_t>(m_warp));
              bulk_commit_group();
            }
            ++blocks_out;
          }
        } else {
          if (!row_ok || n0 >= p.N) return;
          epilogue_store<EPI>(p, g, m, n0, v);
        }
      };
      uint32_t ra[32], rb[32];
      uint4 resa[4], resb[4];
      issue(0, ra, resa);
      tmem_ld_wait(ra);
#pragma unroll 1
      for (int c = 0; c < BN; c += 64) {
        issue(c + 32, rb, resb);
        finish(c, ra, resa);
        __syncwarp();
        tmem_ld_wait(rb);
        if (c + 64 == BN) {
          // Every column of the accumulator is in registers: hand it back to
          // the MMA issuer. The arrival orders only these completed TMEM reads,
          // so it is relaxed and does not wait for this thread's stores.
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty_lead + 8u * static_cast<uint32_t>(acc));
        } else {
          issue(c + 64, ra, resa);
        }
        finish(c + 32, rb, resb);
        if (c + 64 < BN) {
          __syncwarp();
          tmem_ld_wait(ra);
        }
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if constexpr (EPI == kEpiF32Tma || EPI == kEpiGeluTma) {
      if (lane == 0) bulk_wait_group_all();  // every store has left shared memory and landed
      __syncwarp();
    }
  }

  tc_fence_before_sync();
  __syncwarp();
  cluster_sync_all();  // every CTA done: no MMA, copy or remote arrival still targets any of them
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

template <int EPI, int STAGES>
cudaError_t launch_impl(const KParams& kp, cudaStream_t s) {
  using C = PairCfg<STAGES, ksub_of<EPI>()>;
  constexpr size_t kSmem = C::template smem<EPI>();
  constexpr unsigned kCtas = 2;
  auto kern = tc_gemm_pair_kernel<EPI, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // Persistent grid: as many clusters as can be resident at once (per device
  // and per instantiation, since the shared-memory size differs).
  static std::atomic<int> max_clusters[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  int cached = max_clusters[dev].load(std::memory_order_relaxed);
  if (!cached) {
    cfg.gridDim = dim3(kCtas * (num_sms() / kCtas), 1, 1);
    int n = 0;
    cfg.numAttrs = 1;  // the query takes the cluster shape only
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    cfg.numAttrs = 2;
    if (e != cudaSuccess) return e;
    cached = n > 0 ? n : 1;
    max_clusters[dev].store(cached, std::memory_order_relaxed);
  }
  const int clusters = kp.tiles < cached ? kp.tiles : cached;
  cfg.gridDim = dim3(kCtas * clusters, 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, kp);
}

cudaError_t launch_epi(const KParams& kp, int epi, cudaStream_t s) {
  switch (epi) {
    case kEpiGeluBf16:
      return launch_impl<kEpiGeluBf16, stages_of<kEpiGeluBf16>()>(kp, s);
    case kEpiF32:
      return launch_impl<kEpiF32, stages_of<kEpiF32>()>(kp, s);
    case kEpiBwdAct:
      return launch_impl<kEpiBwdAct, stages_of<kEpiBwdAct>()>(kp, s);
    case kEpiF32Tma:
      return launch_impl<kEpiF32Tma, stages_of<kEpiF32Tma>()>(kp, s);
    case kEpiGeluSaveP:
      return launch_impl<kEpiGeluSaveP, stages_of<kEpiGeluSaveP>()>(kp, s);
    case kEpiBf16:
      return launch_impl<kEpiBf16, stages_of<kEpiBf16>()>(kp, s);
    case kEpiGeluTma:
      return launch_impl<kEpiGeluTma, stages_of<kEpiGeluTma>()>(kp, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_pair(const KParams& kp, int epi, cudaStream_t s) { return launch_epi(kp, epi, s); }

}  // namespace tpmlp
