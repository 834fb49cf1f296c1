// gemm_tc.cu — persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// Serves every product of the tensor-parallel MLP in bf16 (X A_i with the
// GeLU fused into the epilogue; H_i B_i as fp32 partials; the shard-ordered
// fused sum; the backward products). One CTA per SM loops over output tiles
// of BM x BN:
//   warp 0, lane 0 : TMA producer — fills a STAGES-deep ring of shared-memory
//                    stages (A box 128 x 64, B box BN x 64, 128-byte swizzle)
//   warp 1         : allocates TMEM; lane 0 issues tcgen05.mma (M=128, N=BN,
//                    K=16 per instruction) into one of two TMEM accumulators
//   warps 2..5     : epilogue — tcgen05.ld the accumulator (warp w reads TMEM
//                    lanes 32*(w%4)..+31 = tile rows), apply the output
//                    treatment and store to global memory
// The two accumulators let the epilogue of tile j overlap the mainloop of
// tile j+1. Every mbarrier wait is bounded; on a timeout the CTA raises an
// abort flag, all roles leave their loops, in-flight copies and MMAs are
// drained and TMEM is freed before the CTA exits.
#include "device.cuh"
#include "internal.h"

#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>

namespace tpmlp {

// Per-device status word: a kernel whose bounded wait ran out of time stores
// the wait's site code here. Read and cleared by read_and_clear_status().
__device__ int g_status = 0;

namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle row of bf16
constexpr int kThreads = 192;

struct KParams {
  CUtensorMap map_a[kMaxGroups];
  CUtensorMap map_b[kMaxGroups];
  void* out[kMaxGroups];
  CUtensorMap map_out[kMaxGroups];  // kEpiF32Tma: fp32 output per group, 32 x 32 boxes, 128-byte swizzle
  const void* aux_p[kMaxGroups];  // kEpiBwdAct: P per group (fp32, row pitch ldo)
  void* aux_ht[kMaxGroups];       // kEpiBwdAct: H^T per group (bf16, row pitch ldt)
  void* aux_dpt[kMaxGroups];      // kEpiBwdAct: dP^T per group (bf16, row pitch ldt)
  int64_t ldo, ldt;
  int M, N;
  int groups;
  int chain;
  int m_blocks, n_blocks, k_blocks;
  int tiles;
  uint64_t wait_ns;
  int inject;
  int group_m;  // tile order: bands of group_m tile rows, rows fastest inside a band (1 = columns fastest)
  int shared;   // kSharedNone / kSharedA / kSharedB: an operand that every group reads
  int stream_out;  // 1: epilogue stores bypass L2 retention (evict-first)
};

template <int BN>
struct Cfg {
  static constexpr int STAGES = BN == 256 ? 4 : 6;
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = BN * BK * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TMEM_COLS = 2 * BN;  // two accumulators
  static constexpr size_t SMEM = 1024 /*alignment slack*/ + size_t(STAGES) * STAGE_BYTES + 256 /*barriers*/;
};

// Maps a tile index to (group, M block, N block). The tiles form a grid of
// `rows` x `cols`, walked in bands of group_m rows with rows fastest inside a
// band, so the tiles in flight together (one per CTA pair) cover about
// group_m rows x (pairs / group_m) columns and each operand panel is fetched
// from DRAM about once per band instead of once per tile.
//   shared A (every group reads the same M x K operand): rows = M blocks,
//     cols = the groups' N blocks side by side;
//   shared B (every group reads the same N x K operand): rows = the groups'
//     M blocks stacked, cols = N blocks;
//   otherwise each group's grid in turn (chain mode: the one output grid).
__device__ __forceinline__ void decode_tile(const KParams& p, int tile, int& g, int& mb, int& nb) {
  int rows_total, cols, base = 0;
  if (p.chain || p.shared == kSharedNone) {
    const int per_group = p.m_blocks * p.n_blocks;
    g = p.chain ? 0 : tile / per_group;
    base = g * per_group;
    rows_total = p.m_blocks;
    cols = p.n_blocks;
  } else if (p.shared == kSharedA) {
    rows_total = p.m_blocks;
    cols = p.groups * p.n_blocks;
  } else {
    rows_total = p.groups * p.m_blocks;
    cols = p.n_blocks;
  }
  const int t = tile - base;
  const int gm = p.group_m > 0 ? p.group_m : 1;
  const int span = gm * cols;
  const int first = (t / span) * gm;
  const int band = min(rows_total - first, gm);
  const int q = t % span;
  const int row = first + q % band;
  const int col = q / band;
  if (p.chain || p.shared == kSharedNone) {
    mb = row;
    nb = col;
  } else if (p.shared == kSharedA) {
    mb = row;
    g = col / p.n_blocks;
    nb = col % p.n_blocks;
  } else {
    g = row / p.m_blocks;
    mb = row % p.m_blocks;
    nb = col;
  }
}

// 16-byte global stores; `stream` marks them evict-first so results that are
// not read again soon do not push the operands out of L2.
__device__ __forceinline__ void store16(void* dst, uint4 v, bool stream) {
  if (stream)
    __stcs(reinterpret_cast<uint4*>(dst), v);
  else
    *reinterpret_cast<uint4*>(dst) = v;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Output treatment of one thread's 32 accumulator columns n0..n0+31 of row m
// (group g). The caller has checked m < M and n0 < N; N is a multiple of 8.
template <int EPI>
__device__ __forceinline__ void epilogue_store(const KParams& p, int g, int64_t m, int n0, const float (&v)[32]) {
  if constexpr (EPI == kEpiGeluBf16) {
    // H = GeLU(acc), bf16, row-major.
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out[g]) + m * p.ldo + n0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (n0 + 8 * j + 8 <= p.N) {
        uint4 w;
        w.x = pack_bf16x2(gelu_fast(v[8 * j + 0]), gelu_fast(v[8 * j + 1]));
        w.y = pack_bf16x2(gelu_fast(v[8 * j + 2]), gelu_fast(v[8 * j + 3]));
        w.z = pack_bf16x2(gelu_fast(v[8 * j + 4]), gelu_fast(v[8 * j + 5]));
        w.w = pack_bf16x2(gelu_fast(v[8 * j + 6]), gelu_fast(v[8 * j + 7]));
        store16(out + 8 * j, w, p.stream_out);
      }
    }
  } else if constexpr (EPI == kEpiF32) {
    float* out = static_cast<float*>(p.out[g]) + m * p.ldo + n0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (n0 + 4 * j + 4 <= p.N)
        store16(out + 4 * j,
                make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]), __float_as_uint(v[4 * j + 2]),
                           __float_as_uint(v[4 * j + 3])),
                p.stream_out);
    }
  } else {
    // Backward activation: acc = dH (row m = token t, column n = feature f).
    // With P from aux_p: dP = dH * GeLU'(P) to out (bf16 [T][ldo]), and the
    // transposes H^T = GeLU(P)^T to aux_ht and dP^T to aux_dpt (bf16 [F][ldt]).
    // The 32 lanes of a warp hold 32 consecutive tokens, so each transposed
    // store of one column is 64 contiguous bytes.
    const float* P = static_cast<const float*>(p.aux_p[g]) + m * p.ldo + n0;
    __nv_bfloat16* dP = static_cast<__nv_bfloat16*>(p.out[g]) + m * p.ldo + n0;
    __nv_bfloat16* Ht = static_cast<__nv_bfloat16*>(p.aux_ht[g]) + int64_t(n0) * p.ldt + m;
    __nv_bfloat16* dPt = static_cast<__nv_bfloat16*>(p.aux_dpt[g]) + int64_t(n0) * p.ldt + m;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (n0 + 8 * j + 8 > p.N) continue;
      const float4 p0 = *reinterpret_cast<const float4*>(P + 8 * j);
      const float4 p1 = *reinterpret_cast<const float4*>(P + 8 * j + 4);
      const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
      float h[8], d[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float gv, dg;
        gelu_and_grad_fast(pv[e], gv, dg);
        h[e] = gv;
        d[e] = v[8 * j + e] * dg;
      }
      uint4 w;
      w.x = pack_bf16x2(d[0], d[1]);
      w.y = pack_bf16x2(d[2], d[3]);
      w.z = pack_bf16x2(d[4], d[5]);
      w.w = pack_bf16x2(d[6], d[7]);
      store16(dP + 8 * j, w, false);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int64_t o = int64_t(8 * j + e) * p.ldt;
        Ht[o] = __float2bfloat16_rn(h[e]);
        dPt[o] = __float2bfloat16_rn(d[e]);
      }
    }
  }
}

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
  const WaitGuard guard{abort_flag, p.wait_ns, &g_status};
  const int kb_per_tile = p.chain ? p.groups * p.k_blocks : p.k_blocks;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, parity_bits = 0;
      int fill = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
        int g, mb, nb;
        decode_tile(p, tile, g, mb, nb);
        int gg = g, kk = 0;  // group and K block of the next fill (chain mode walks the groups in order)
        for (int kb = 0; kb < kb_per_tile; ++kb, ++kk) {
          if (kk == p.k_blocks) {
            kk = 0;
            ++gg;
          }
          if (!wait_bounded(empty + stage, phase ^ 1u, guard, kSiteProducer)) {
            ok = false;
            break;
          }
          ++fill;
          if (fill != p.inject) {
            mbar_arrive_expect_tx(full + stage, C::STAGE_BYTES);
            tma_load_2d(sA + stage * C::A_BYTES, &p.map_a[gg], kk * BK, mb * BM, full + stage);
            tma_load_2d(sB + stage * C::B_BYTES, &p.map_b[gg], kk * BK, nb * BN, full + stage);
            issued |= 1u << stage;
            parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
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
      constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
        if (!wait_bounded(acc_empty + acc, acc_phase ^ 1u, guard, kSiteMmaAcc)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < kb_per_tile; ++kb) {
          if (!wait_bounded(full + stage, phase, guard, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a0 = smem_addr(sA + stage * C::A_BYTES);
          const uint32_t b0 = smem_addr(sB + stage * C::B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            tc_mma_bf16(d_tmem, smem_desc_sw128(a0 + 32u * k), smem_desc_sw128(b0 + 32u * k), IDESC,
                        (kb | k) != 0 ? 1u : 0u);
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
      bool ok = wait_bounded(acc_full + acc, acc_phase, guard, kSiteEpilogue);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after_sync();
      const int64_t m = int64_t(mb) * BM + row;
      const bool row_ok = m < p.M;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        float v[32];
        __syncwarp();  // tcgen05.ld is warp-collective
        tmem_ld_32cols(t_row + static_cast<uint32_t>(c), v);
        if (c + 32 == BN) {
          tc_fence_before_sync();
          mbar_arrive(acc_empty + acc);  // accumulator may be overwritten now
        }
        const int n0 = nb * BN + c;
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

// ============================================================================
// CTA-pair variant (tcgen05 cta_group::2): a cluster of two CTAs on two SMs
// computes one 256 x 256 tile. Each CTA loads its own 128 rows of the M x K
// operand and its own 128 of the 256 rows of the N x K operand; the even CTA
// issues M=256, N=256 MMAs that read both CTAs' shared memory and write each
// CTA's TMEM (its 128 rows x 256 fp32 columns). Per SM this moves half the
// N x K operand bytes of the single-CTA kernel for the same MMA work.
//   both CTAs, warp 0 lane 0 : TMA producer for the CTA's halves; completion is
//                              counted on the even CTA's full barrier, which
//                              the even producer arms with both CTAs' bytes
//   even CTA, warp 1 lane 0  : MMA issuer; commits free each stage and publish
//                              each accumulator in BOTH CTAs (multicast)
//   both CTAs, warps 2..5    : epilogue of the CTA's own 128 rows; release the
//                              accumulator by arriving on the even CTA's barrier
// ============================================================================

template <int STAGES_>
struct PairCfg {
  static constexpr int STAGES = STAGES_;
  static constexpr uint32_t A_BYTES = 128 * BK * 2;  // this CTA's 128 rows
  static constexpr uint32_t B_BYTES = 128 * BK * 2;  // this CTA's half of the 256 N rows
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TMEM_COLS = 512;  // two accumulators of 256 fp32 columns
  // kEpiF32Tma: two 32 x 32 fp32 staging blocks (4 KB each) per epilogue warp.
  static constexpr uint32_t OUT_BLOCK = 32 * 32 * 4;
  template <int EPI>
  static constexpr uint32_t staging() {
    return EPI == kEpiF32Tma ? 4 * 2 * OUT_BLOCK : 0;
  }
  template <int EPI>
  static constexpr size_t smem() { return 1024 + size_t(STAGES) * STAGE_BYTES + staging<EPI>() + 256; }
};

template <int EPI, int STAGES>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_pair_kernel(const __grid_constant__ KParams p) {
  using C = PairCfg<STAGES>;
  constexpr int BN = 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  uint8_t* s_out = smem + C::STAGES * C::STAGE_BYTES;  // 1024-aligned staging of kEpiF32Tma
  uint64_t* full = reinterpret_cast<uint64_t*>(s_out + C::template staging<EPI>());
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 = even CTA (issues the MMAs), 1 = odd
  const int cluster = static_cast<int>(cluster_id_x());
  const int nclusters = static_cast<int>(cluster_count_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full + s, 1);   // even CTA: its producer's arrive (+ both CTAs' bytes)
      mbar_init(empty + s, 1);  // one multicast commit per use
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full + b, 1);   // one multicast commit per tile
      mbar_init(acc_empty + b, 8);  // even CTA: one arrival per epilogue warp of both CTAs
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
  cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const WaitGuard guard{abort_flag, p.wait_ns, &g_status};
  const uint32_t peer_abort = map_to_cta(smem_addr(const_cast<int*>(abort_flag)), rank ^ 1u);
  const int kb_per_tile = p.chain ? p.groups * p.k_blocks : p.k_blocks;
  bool aborted = false;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, parity_bits = 0;
      int fill = 0;
      for (int tile = cluster; !aborted && tile < p.tiles; tile += nclusters) {
        int g, mb, nb;
        decode_tile(p, tile, g, mb, nb);
        const int m0 = mb * 256 + static_cast<int>(rank) * 128;
        const int n0 = nb * BN + static_cast<int>(rank) * 128;
        int gg = g, kk = 0;  // group and K block of the next fill (chain mode walks the groups in order)
        for (int kb = 0; kb < kb_per_tile; ++kb, ++kk) {
          if (kk == p.k_blocks) {
            kk = 0;
            ++gg;
          }
          if (!wait_bounded(empty + stage, phase ^ 1u, guard, kSiteProducer)) {
            aborted = true;
            break;
          }
          const uint32_t full_even = map_to_cta(smem_addr(full + stage), 0);
          ++fill;
          if (fill != p.inject) {
            if (rank == 0) {
              mbar_arrive_expect_tx(full + stage, 2 * C::STAGE_BYTES);
              armed |= 1u << stage;
              parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
            }
            tma_load_2d_pair(sA + stage * C::A_BYTES, &p.map_a[gg], kk * BK, m0, full_even);
            tma_load_2d_pair(sB + stage * C::B_BYTES, &p.map_b[gg], kk * BK, n0, full_even);
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (aborted) {
        st_cluster_u32(peer_abort, 1u);
        if (rank == 0) {
          for (int s = 0; s < C::STAGES; ++s)
            if (armed >> s & 1u) wait_drain(full + s, (parity_bits >> s) & 1u, p.wait_ns);
        } else {
          // The odd CTA's copies are counted on the even CTA's barriers; give
          // any copy still in flight time to land before shared memory is released.
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 200000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (even CTA)
      constexpr uint32_t IDESC = idesc_bf16_f32(256, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int tile = cluster; !aborted && tile < p.tiles; tile += nclusters) {
        if (!wait_bounded(acc_empty + acc, acc_phase ^ 1u, guard, kSiteMmaAcc)) {
          aborted = true;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < kb_per_tile; ++kb) {
          if (!wait_bounded(full + stage, phase, guard, kSiteMmaFull)) {
            aborted = true;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a0 = smem_addr(sA + stage * C::A_BYTES);
          const uint32_t b0 = smem_addr(sB + stage * C::B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            tc_mma_bf16_pair(d_tmem, smem_desc_sw128(a0 + 32u * k), smem_desc_sw128(b0 + 32u * k), IDESC,
                             (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit_pair_multicast(empty + stage, 0x3);  // frees stage `stage` in both CTAs
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (aborted) break;
        tc_commit_pair_multicast(acc_full + acc, 0x3);  // accumulator complete in both CTAs
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (aborted) {
        st_cluster_u32(peer_abort, 1u);
        tc_commit_pair_multicast(drain, 0x1);
        wait_drain(drain, 0, p.wait_ns);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5 of both CTAs)
    const int quarter = warp & 3;  // rows quarter*32 .. +31 of this CTA's 128 (its TMEM lane quarter)
    const uint32_t acc_empty_even0 = map_to_cta(smem_addr(acc_empty), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    int blocks_out = 0;  // kEpiF32Tma: 32 x 32 blocks this warp has handed to TMA so far
    for (int tile = cluster; tile < p.tiles; tile += nclusters) {
      int g, mb, nb;
      decode_tile(p, tile, g, mb, nb);
      bool ok = wait_bounded(acc_full + acc, acc_phase, guard, kSiteEpilogue);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) st_cluster_u32(peer_abort, 1u);
        break;
      }
      tc_fence_after_sync();
      const int64_t m_warp = int64_t(mb) * 256 + int64_t(rank) * 128 + quarter * 32;  // row of lane 0
      const int64_t m = m_warp + lane;
      const bool row_ok = m < p.M;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        float v[32];
        __syncwarp();
        tmem_ld_32cols(t_row + static_cast<uint32_t>(c), v);
        if (c + 32 == BN) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(acc_empty_even0 + 8u * static_cast<uint32_t>(acc));
        }
        const int n0 = nb * BN + c;
        if constexpr (EPI == kEpiF32Tma) {
          // Stage the warp's 32 x 32 fp32 block in shared memory with the
          // 128-byte swizzle (16-byte chunk j of row r at slot j ^ (r % 8),
          // conflict-free for these row-per-lane writes), then one TMA store
          // writes it as whole 128-byte lines, clipped to M x N.
          if (n0 >= p.N || m_warp >= p.M) continue;  // warp-uniform
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
            tma_store_2d(&p.map_out[g], buf, n0, static_cast<int32_t>(m_warp));
            bulk_commit_group();
          }
          ++blocks_out;
        } else {
          if (!row_ok || n0 >= p.N) continue;
          epilogue_store<EPI>(p, g, m, n0, v);
        }
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if constexpr (EPI == kEpiF32Tma) {
      if (lane == 0) bulk_wait_group_all();  // every store has left shared memory and landed
      __syncwarp();
    }
  }

  tc_fence_before_sync();
  __syncwarp();
  cluster_sync_all();  // both CTAs done: no MMA, copy or remote arrival still targets either CTA
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

template <int EPI, int STAGES>
cudaError_t launch_pair_impl(const KParams& kp, cudaStream_t s) {
  using C = PairCfg<STAGES>;
  constexpr size_t kSmem = C::template smem<EPI>();
  auto kern = tc_gemm_pair_kernel<EPI, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Persistent grid: as many CTA pairs as can be resident at once (per device
  // and per instantiation, since the shared-memory size differs).
  static int max_pairs[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  int& cached = max_pairs[dev];
  if (!cached) {
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    cached = n > 0 ? n : 1;
  }
  const int pairs = kp.tiles < cached ? kp.tiles : cached;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, kp);
}

template <int BN, int EPI>
cudaError_t launch_impl(const KParams& kp, cudaStream_t s) {
  using C = Cfg<BN>;
  auto kern = tc_gemm_kernel<BN, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::SMEM));
  if (e != cudaSuccess) return e;
  const int grid = kp.tiles < num_sms() ? kp.tiles : num_sms();
  kern<<<grid, kThreads, C::SMEM, s>>>(kp);
  return cudaGetLastError();
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

}  // namespace

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

static int env_int(const char* name, int dflt) {
  const char* e = getenv(name);
  return e && *e ? atoi(e) : dflt;
}

// The CTA-pair kernel is the default; TPMLP_TC_PAIR=0 selects the
// single-CTA kernel (read once per process; kept for comparisons).
static bool use_pair_kernel() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("TPMLP_TC_PAIR");
    v = (e && e[0] == '0') ? 0 : 1;
  }
  return v == 1;
}

int tc_box_rows_b(int N) {
  if (use_pair_kernel()) return 128;  // each CTA of a pair loads half of the 256 N rows
  return N <= 128 ? 128 : 256;
}

// A 2-D row-major tensor [rows, cols] with a row pitch of pitch_bytes, boxes
// of box_cols x box_rows elements, 128-byte swizzle.
static bool encode_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, int64_t rows, int64_t cols,
                      int64_t pitch_bytes, int box_cols, int box_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
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

bool make_output_map_f32(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t pitch_elems) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, rows, cols, pitch_elems * 4, 32, 32);
}


cudaError_t launch_tc_gemm(const TcGemm& g, uint64_t wait_ns, cudaStream_t s) {
  KParams kp;
  memset(&kp, 0, sizeof(kp));
  for (int i = 0; i < g.groups; ++i) {
    kp.map_a[i] = *g.map_a[i];
    kp.map_b[i] = *g.map_b[i];
    kp.out[i] = g.out[i];
    kp.aux_p[i] = g.aux_p[i];
    kp.aux_ht[i] = g.aux_ht[i];
    kp.aux_dpt[i] = g.aux_dpt[i];
    if (g.map_out[i]) kp.map_out[i] = *g.map_out[i];
  }
  // CTA pairs with 256 x 256 tiles, unless the product has too few of those
  // tiles to occupy a quarter of the SMs: then single CTAs with 128-row tiles
  // (and 128-column tiles, the operand boxes that pair mode encodes) spread it
  // over four times as many SMs.
  const int pair_tiles = ((g.M + 255) / 256) * ((g.N + 255) / 256) * (g.chain ? 1 : g.groups);
  const bool pair = use_pair_kernel() && pair_tiles >= num_sms() / 4;
  // Outputs with TMA maps leave the pair kernel through TMA stores.
  const bool tma_out = pair && g.map_out[0] != nullptr && env_int("TPMLP_TMA_STORE", 1) != 0;
  const int BN = pair ? 256 : tc_box_rows_b(g.N);
  const int TM = pair ? 256 : BM;
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
  kp.inject = g.inject;
  kp.group_m = env_int("TPMLP_GROUP_M", g.group_m);
  kp.shared = g.shared;
  kp.stream_out = env_int("TPMLP_STREAM_OUT", g.stream_out);
  if (kp.tiles == 0) return cudaSuccess;
  switch (g.epi) {
    case kEpiGeluBf16:
      return pair ? launch_pair_impl<kEpiGeluBf16, 6>(kp, s)
                  : (BN == 256 ? launch_impl<256, kEpiGeluBf16>(kp, s) : launch_impl<128, kEpiGeluBf16>(kp, s));
    case kEpiF32:
      if (tma_out) return launch_pair_impl<kEpiF32Tma, 6>(kp, s);
      return pair ? launch_pair_impl<kEpiF32, 6>(kp, s)
                  : (BN == 256 ? launch_impl<256, kEpiF32>(kp, s) : launch_impl<128, kEpiF32>(kp, s));
    case kEpiBwdAct:
      return pair ? launch_pair_impl<kEpiBwdAct, 6>(kp, s)
                  : (BN == 256 ? launch_impl<256, kEpiBwdAct>(kp, s) : launch_impl<128, kEpiBwdAct>(kp, s));
    default:
      return cudaErrorInvalidValue;
  }
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = v > 0 ? v : 1;
  }
  return cached[dev];
}

}  // namespace tpmlp
