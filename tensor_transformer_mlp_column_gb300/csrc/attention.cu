// attention.cu — the local attention of head-split tensor parallelism
// (duoan.github.io "Tensor Parallelism in Megatron-LM", §4): for every
// sequence b and head h of every rank, O = softmax(Q K^T / sqrt(d_h)) V with
// no mask, reading Q, K from the rank's QKV projection [T, 3 D/n] and V from
// its transpose V^T [D/n, T], and writing O into the rank's [T, D/n] block.
//
// Exact tensor-core kernel (bf16, d_h = 64, seq <= 512, seq % 8 == 0): one
// CTA of 16 warps per (128-query tile, head, sequence).
//   thread 0 : TMA-loads the Q tile, all keys and all of V^T for the head
//              into 128-byte-swizzled shared memory (one mbarrier), then
//              issues S = Q K^T (M=128, N=128 per key block, K=16 steps)
//              into tensor memory: the whole score row, up to 512 columns
//   16 warps : warp w reads TMEM lanes 32 (w % 4) .. (its query rows) and
//              column quarter w / 4 of the scores: one pass for the maximum,
//              a second for p = 2^((s - max) * log2(e) / sqrt(d_h)) and its
//              fp32 sum, writing p as bf16 into shared memory in the
//              128-byte-swizzled K-major layout of an MMA operand (chunks
//              4..7 reuse the key buffer, dead once S is computed); the four
//              quarters' maxima and sums meet in shared memory. Then
//              O = P V (M=128, N=64, one chunk of 64 keys per 4 MMAs) into
//              TMEM columns 0..63, and O / sum rounded to bf16, each warp
//              writing 16 of the 64 columns of its rows.
// The softmax is exact (the full row is in tensor memory), not the running
// rescale of a streaming kernel. Every wait is bounded; on a timeout the CTA
// records the site, drains its copies and MMAs and frees its tensor memory.
//
// fp32 kernel (any d_h <= 128, seq <= 8192): one warp per query row, scores
// in shared memory, the same two passes, on the CUDA cores.
#include <cstdlib>

#include "device.cuh"
#include "internal.h"

namespace tpmlp {

namespace {

constexpr int kAttnThreads = 512;  // 16 warps: 4 TMEM lane quarters x 4 column groups
constexpr int kF32Threads = 128;   // fp32 kernel: 4 warps, one query row each
constexpr uint32_t kQBytes = 128 * 128;       // 128 query rows x 64 bf16
constexpr uint32_t kKBlockBytes = 128 * 128;  // 128 key rows x 64 bf16
constexpr uint32_t kVtChunkBytes = 64 * 128;  // 64 d-rows x 64 keys
constexpr uint32_t kPChunkBytes = 128 * 128;  // 128 query rows x 64 keys
constexpr int kPhaseChunks = 4;               // P chunks in the P buffer; the rest reuse the key buffer

struct AttnParams {
  CUtensorMap map_qkv[kMaxGroups];  // QKV_i [T, 3 Dn] bf16, boxes 64 x 128
  CUtensorMap map_vt[kMaxGroups];   // V_i^T [Dn, T] bf16 (row pitch T8), boxes 64 x 64
  void* out[kMaxGroups];            // O_i [T, Dn]
  int seq, Dn, local_heads;
  int q_tiles, heads, items;  // streaming kernel: query tiles per head, heads of all ranks, work items
  float scale_log2;  // log2(e) / sqrt(d_h)
  uint64_t wait_ns;
  int* status;
};

__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__host__ __device__ constexpr uint32_t attn_smem_bytes(int nkv, int nch) {
  return 1024 + kQBytes + uint32_t(nkv) * kKBlockBytes + uint32_t(nch) * kVtChunkBytes +
         uint32_t(nch < kPhaseChunks ? nch : kPhaseChunks) * kPChunkBytes + 2 * 4 * 128 * 4 + 64;
}

// 16 consecutive 32-bit TMEM columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 2^x on the special-function unit (relative error about 2^-22, flushes
// subnormal results to zero), used for the softmax weights, which are rounded
// to bf16 afterwards.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed pairs of fp32 (sm_100 and later): one instruction for two lanes'
// worth of fused multiply-add or add.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t d, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(d));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Shared-memory address of P chunk c (64 keys x 128 query rows): chunks 0..3
// in the P buffer, chunks 4..7 in the key buffer, free once S is computed.
__device__ __forceinline__ uint8_t* p_chunk(uint8_t* sP, uint8_t* sK, int c) {
  return c < kPhaseChunks ? sP + c * kPChunkBytes : sK + (c - kPhaseChunks) * kPChunkBytes;
}

__global__ void __launch_bounds__(kAttnThreads, 1) attn_tc_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nkv = (p.seq + 127) / 128;  // key blocks of the score product
  const int nch = (p.seq + 63) / 64;    // 64-key chunks of P and V^T
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + kQBytes;
  uint8_t* sVt = sK + nkv * kKBlockBytes;
  uint8_t* sP = sVt + nch * kVtChunkBytes;
  float* red_max = reinterpret_cast<float*>(sP + (nch < kPhaseChunks ? nch : kPhaseChunks) * kPChunkBytes);  // [4][128]
  float* red_sum = red_max + 4 * 128;                                                                         // [4][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(red_sum + 4 * 128);
  uint64_t* bar_load = bars;      // Q and the keys
  uint64_t* bar_mma = bars + 1;
  uint64_t* bar_drain = bars + 2;
  uint64_t* bar_v = bars + 3;      // V^T, needed only by the P V product
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 5);

  const int qt = blockIdx.x, gh = blockIdx.y, b = blockIdx.z;
  const int shard = gh / p.local_heads, hl = gh % p.local_heads;
  // Debug build: the CTA's query tile, rank and output must exist (CTA-uniform).
  if (!TPMLP_DCHECK(qt * 128 < p.seq && shard < kMaxGroups && p.out[shard] != nullptr,
                    threadIdx.x == 0 ? p.status : nullptr, kChkAttnTile))
    return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3;      // TMEM lanes (= query rows) 32*quarter .. +31
  const int cgroup = warp >> 2;      // column group 0..3 of the score row
  const int row = quarter * 32 + lane;
  const uint32_t tmem_cols = nkv <= 1 ? 128u : (nkv <= 2 ? 256u : 512u);

  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_drain, 1);
    mbar_init(bar_v, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, tmem_cols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // set-up done: wait for the kernel that wrote Q, K and V
  pdl_launch_dependents();
  const WaitGuard guard{abort_flag, p.wait_ns, p.status};

  const int32_t row0 = b * p.seq;  // first token of the sequence
  if (tid == 0) {
    const CUtensorMap* mq = &p.map_qkv[shard];
    const CUtensorMap* mv = &p.map_vt[shard];
    mbar_arrive_expect_tx(bar_load, kQBytes + nkv * kKBlockBytes);
    tma_load_2d(sQ, mq, hl * 64, row0 + qt * 128, bar_load);
    for (int j = 0; j < nkv; ++j) tma_load_2d(sK + j * kKBlockBytes, mq, p.Dn + hl * 64, row0 + j * 128, bar_load);
    mbar_arrive_expect_tx(bar_v, nch * kVtChunkBytes);
    for (int c = 0; c < nch; ++c) tma_load_2d(sVt + c * kVtChunkBytes, mv, row0 + c * 64, hl * 64, bar_v);
  }
  bool ok = wait_bounded(bar_load, 0, guard, kSiteProducer);
  if (ok && tid == 0) {
    tc_fence_after_sync();
    const uint64_t dq = smem_desc_sw128(smem_addr(sQ));
    constexpr uint32_t kIdS = idesc_bf16_f32(128, 128);
    for (int j = 0; j < nkv; ++j) {
      const uint64_t dk = smem_desc_sw128(smem_addr(sK + j * kKBlockBytes));
#pragma unroll
      for (int k = 0; k < 4; ++k) tc_mma_bf16(tmem + j * 128, dq + 2 * k, dk + 2 * k, kIdS, k > 0 ? 1u : 0u);
    }
    tc_commit(bar_mma);
  }
  ok = ok && wait_bounded(bar_mma, 0, guard, kSiteMmaFull);

  // ---- softmax: warp (quarter, cgroup) owns rows 32*quarter.. and a quarter
  // of the score columns; the row's maximum and sum combine the four groups.
  tc_fence_after_sync();
  const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  const int gcols = nkv * 32;  // columns per group (a multiple of 32)
  const int col0 = cgroup * gcols;
  float mx = -INFINITY;
  if (ok) {
    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // independent chains
    for (int g = 0; g < gcols; g += 32) {
      float v[32];
      tmem_ld_32cols(t_row + col0 + g, v);
      if (col0 + g + 32 <= p.seq) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) m4[(j >> 1) & 3] = fmax3(m4[(j >> 1) & 3], v[j], v[j + 1]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col0 + g + j < p.seq) m4[j & 3] = fmaxf(m4[j & 3], v[j]);
      }
    }
    mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
  }
  red_max[cgroup * 128 + row] = mx;
  __syncthreads();
  mx = fmaxf(fmaxf(red_max[row], red_max[128 + row]), fmaxf(red_max[256 + row], red_max[384 + row]));
  const float mb = mx * p.scale_log2;
  float sum = 0.f;
  if (ok) {
    for (int g = 0; g < gcols; g += 32) {
      const int col = col0 + g;  // first of 32 columns: half (col % 64) / 32 of chunk col / 64
      if (col >= nch * 64) break;
      float v[32];
      tmem_ld_32cols(t_row + col, v);
      uint32_t w[16];
      float s2[2] = {0.f, 0.f};
      if (col + 32 <= p.seq) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float e0 = ex2_approx(fmaf(v[j], p.scale_log2, -mb));
          const float e1 = ex2_approx(fmaf(v[j + 1], p.scale_log2, -mb));
          s2[0] += e0;
          s2[1] += e1;
          w[j / 2] = pack2_bf16(e0, e1);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float e0 = col + j < p.seq ? ex2_approx(fmaf(v[j], p.scale_log2, -mb)) : 0.f;
          const float e1 = col + j + 1 < p.seq ? ex2_approx(fmaf(v[j + 1], p.scale_log2, -mb)) : 0.f;
          s2[0] += e0;
          s2[1] += e1;
          w[j / 2] = pack2_bf16(e0, e1);
        }
      }
      sum += s2[0] + s2[1];
      uint8_t* prow = p_chunk(sP, sK, col / 64) + row * 128;
      const int half = (col % 64) / 32;
      // 16-byte unit u of a 128-byte row r sits at unit u ^ (r % 8).
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(prow + (((half * 4 + q) ^ (row & 7)) << 4)) =
            make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
  }
  red_sum[cgroup * 128 + row] = sum;
  fence_proxy_async_smem();  // P, written by threads, is read by the tensor cores
  tc_fence_before_sync();
  __syncthreads();
  if (tid == 0 && ok && !*abort_flag && wait_bounded(bar_v, 0, guard, kSiteProducer)) {
    tc_fence_after_sync();
    constexpr uint32_t kIdO = idesc_bf16_f32(128, 64);
    for (int c = 0; c < nch; ++c) {
      const uint64_t dp = smem_desc_sw128(smem_addr(p_chunk(sP, sK, c)));
      const uint64_t dv = smem_desc_sw128(smem_addr(sVt + c * kVtChunkBytes));
#pragma unroll
      for (int k = 0; k < 4; ++k) tc_mma_bf16(tmem, dp + 2 * k, dv + 2 * k, kIdO, (c > 0 || k > 0) ? 1u : 0u);
    }
    tc_commit(bar_mma);
  }
  ok = ok && !*abort_flag && wait_bounded(bar_mma, 1, guard, kSiteEpilogue);

  // ---- O / sum -> bf16: warp (quarter, cgroup) writes columns 16*cgroup .. +15 of its rows
  if (ok) {
    tc_fence_after_sync();
    float o[16];
    tmem_ld_16cols(t_row + cgroup * 16, o);
    const int qi = qt * 128 + row;
    if (qi < p.seq) {
      const float inv = 1.0f / (((red_sum[row] + red_sum[128 + row]) + red_sum[256 + row]) + red_sum[384 + row]);
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out[shard]) + (static_cast<int64_t>(row0) + qi) * p.Dn +
                           hl * 64 + cgroup * 16;
      reinterpret_cast<uint4*>(dst)[0] =
          make_uint4(pack2_bf16(o[0] * inv, o[1] * inv), pack2_bf16(o[2] * inv, o[3] * inv),
                     pack2_bf16(o[4] * inv, o[5] * inv), pack2_bf16(o[6] * inv, o[7] * inv));
      reinterpret_cast<uint4*>(dst)[1] =
          make_uint4(pack2_bf16(o[8] * inv, o[9] * inv), pack2_bf16(o[10] * inv, o[11] * inv),
                     pack2_bf16(o[12] * inv, o[13] * inv), pack2_bf16(o[14] * inv, o[15] * inv));
    }
  }

  // ---- clean-up: after an abort, let copies and products in flight finish first
  __syncthreads();
  if (*abort_flag && tid == 0) {
    wait_drain(bar_load, 0, p.wait_ns);
    wait_drain(bar_v, 0, p.wait_ns);
    tc_commit(bar_drain);
    wait_drain(bar_drain, 0, p.wait_ns);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// ------------------------------------------------------------------ streaming form (any seq)
//
// CTAs of 8 softmax warps, an MMA warp and a load warp, 112 KB of shared
// memory and 256 TMEM columns, so two CTAs share an SM and one's loads and
// products overlap the other's softmax. The work items (128-query tile, head,
// sequence) go to a persistent grid of two CTAs per SM, each running its
// items through one pipeline: the ring runs on from item to item, an item's
// Q lands once the previous item's last score product has read the buffer,
// and its first P V product waits until the previous item's O is in the
// softmax warps' registers (6-8 % faster at seq 512 than a CTA per item, 1-3 %
// at 1024-4096). Keys go in blocks of 128 with a running maximum m and sum l
// per query row:
//   load thread: Q once, then K_j and V_j^T (16 KB each) through a ring of
//     two slots in the order the products read them (K_0, then K_j, V_{j-1}
//     for j = 1.., then the last V), each slot refilled as soon as the product
//     that read it has finished.
//   MMA thread: S_j = Q K_j^T into TMEM columns 0..127 once every softmax warp
//     holds S_{j-1} in registers, then P_{j-1} V_{j-1} accumulated into O
//     (TMEM columns 128..255) once the softmax has written P_{j-1}; every
//     wait bounded. P has two buffers, block j using buffer j % 2, so the
//     softmax writes P_j as soon as P_{j-2} V_{j-2} has finished and waits
//     for P_{j-1} V_{j-1} only before it rescales O.
//   softmax warp w: TMEM lanes 32 (w % 4) (its query rows) and key half w / 4
//     of the block, with a running maximum, row sum and output accumulator
//     O_half of its own: new running maximum m' (moved only when the block's
//     maximum exceeds m by more than 2^8 in weight), a = 2^((m - m') log2(e)/sqrt(d_h)),
//     p = 2^((s - m') log2(e)/sqrt(d_h)) written as bf16 into the swizzled P
//     operand, l <- a l + sum p, and O_half <- a O_half in TMEM when the
//     maximum moved.
// (A one-CTA-per-SM form with every buffer doubled and 16 softmax warps was
// measured slower: 217 vs 186 us at seq 4096; two independent CTAs per SM
// overlap better than 16 warps meeting at a barrier every block.)
// At the end the two halves of a row merge and O / l is rounded to bf16. The
// same result as the exact kernel up to rounding (the weights of earlier
// blocks are rescaled in fp32).

constexpr int kStrmSoftmaxWarps = 8;
constexpr int kStrmThreads = (kStrmSoftmaxWarps + 2) * 32;  // + the MMA warp and the load warp
constexpr uint32_t kStrmSlotBytes = 128 * 128;              // K of 128 keys (128 x 64 bf16) or their V^T (64 x 128)
constexpr int kStrmSlots = 2;
constexpr uint32_t kStrmPBufBytes = 2 * kPChunkBytes;  // P of 128 keys
constexpr uint32_t kStrmPBytes = 2 * kStrmPBufBytes;   // two P buffers, blocks alternating
// No alignment slack: the dynamic shared memory is declared 1024-aligned (and
// checked), so two CTAs fit an SM with both P buffers.
constexpr uint32_t kStrmSmem = kQBytes + kStrmSlots * kStrmSlotBytes + kStrmPBytes + 256;
static_assert(2 * kVtChunkBytes == kStrmSlotBytes, "V^T of a key block fills one ring slot");

// 32 TMEM columns of this warp's lanes without waiting: the registers are valid
// only after tmem_wait_ld(), so several loads can be in flight at once.
__device__ __forceinline__ void tmem_ld_32cols_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st_32cols(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kStrmThreads, 2) attn_stream_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_addr(smem_raw) & 1023u) {  // the 128-byte-swizzled operands need 1024-byte alignment
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kSiteSmemAlign);
    return;  // CTA-uniform, before any barrier or TMEM allocation
  }
  uint8_t* smem = smem_raw;
  uint8_t* sQ = smem;
  uint8_t* sRing = sQ + kQBytes;  // kStrmSlots slots of one K or V^T block
  uint8_t* sP = sRing + kStrmSlots * kStrmSlotBytes;  // two buffers of kStrmPBufBytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + kStrmPBytes);
  uint64_t* bar_q = bars + 0;                     // the item's Q has landed (phase = item count)
  uint64_t* ring_full = bars + 1;                 // [kStrmSlots]
  uint64_t* ring_empty = bars + 1 + kStrmSlots;   // [kStrmSlots]: the product that read the slot has finished
  uint64_t* s_full = bars + 1 + 2 * kStrmSlots;
  // [2]: one arrival per softmax warp once P_k is written and O rescaled, k
  // even / odd (phase k / 2 of s_free[k % 2]). Two barriers because a warp
  // may finish block k+1 (it waits only for P_{k-1} V_{k-1}) before the MMA
  // thread has waited for block k: one barrier could then be two phases
  // ahead of that wait. Block indices k count on across the CTA's items.
  uint64_t* s_free = s_full + 1;
  uint64_t* x_bar = s_full + 3;   // one arrival per softmax warp: the halves' partial maxima (sums) written
  uint64_t* drain = s_full + 4;
  uint64_t* s_read = s_full + 5;  // one arrival per softmax warp: its S columns are in registers
  uint64_t* o_done = s_full + 6;  // [2]: P_k V_k done, k even / odd (phase k / 2 of o_done[k % 2])
  uint64_t* q_free = s_full + 8;  // the item's last score product has finished reading Q
  uint64_t* o_read = s_full + 9;  // one arrival per softmax warp: the item's O is in registers
  volatile int* abort_flag = reinterpret_cast<volatile int*>(s_full + 10);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + 11);

  const int nkv = (p.seq + 127) / 128;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr uint32_t kCols = 256;  // S: columns 0..127; O_0, O_1 (the two key halves): 128..191, 192..255
  constexpr int kMmaWarp = kStrmSoftmaxWarps, kLoadWarp = kStrmSoftmaxWarps + 1;
  // Item i of the launch: query tile i % q_tiles of head (i / q_tiles) % heads
  // of sequence i / (q_tiles * heads), so that items taken together share
  // their keys and values. The CTA takes items blockIdx.x, + gridDim.x, ...
  struct Item {
    int qt, shard, hl;
    int32_t row0;
  };
  auto decode = [&](int i, Item& it) {
    it.qt = i % p.q_tiles;
    const int r = i / p.q_tiles;
    const int gh = r % p.heads;
    it.shard = gh / p.local_heads;
    it.hl = gh % p.local_heads;
    it.row0 = (r / p.heads) * p.seq;
    // Debug build: the item's query tile, rank and output exist (the same
    // answer in every role, so all of them skip a bad item alike).
    return TPMLP_DCHECK(it.qt * 128 < p.seq && it.shard < kMaxGroups && p.out[it.shard] != nullptr,
                        tid == 0 ? p.status : nullptr, kChkAttnTile);
  };

  if (tid == 0) {
    mbar_init(bar_q, 1);
    for (int i = 0; i < kStrmSlots; ++i) {
      mbar_init(ring_full + i, 1);
      mbar_init(ring_empty + i, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, kStrmSoftmaxWarps);
    mbar_init(s_free + 1, kStrmSoftmaxWarps);
    mbar_init(s_read, kStrmSoftmaxWarps);
    mbar_init(o_done, 1);
    mbar_init(o_done + 1, 1);
    mbar_init(x_bar, kStrmSoftmaxWarps);
    mbar_init(drain, 1);
    mbar_init(q_free, 1);
    mbar_init(o_read, kStrmSoftmaxWarps);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, kCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // set-up done: wait for the kernel that wrote Q, K and V
  pdl_launch_dependents();
  const uint32_t tS = tmem, tO = tmem + 128;
  const WaitGuard guard{abort_flag, p.wait_ns, p.status};

  if (warp == kLoadWarp) {
    if (lane == 0) {
      // ---------------- loads: per item Q (once the previous item's last
      // score product has read the buffer), then the ring in the order the
      // products read it; the ring runs on from item to item.
      int n = 0;  // ring position of the next load
      int k = 0;  // items done by this CTA
      bool ok = true;
      for (int i = blockIdx.x; ok && i < p.items; i += gridDim.x) {
        Item it;
        if (!decode(i, it)) continue;
        const CUtensorMap* mq = &p.map_qkv[it.shard];
        const CUtensorMap* mv = &p.map_vt[it.shard];
        const int kx = p.Dn + it.hl * 64;
        if (k > 0 && !wait_bounded(q_free, (k - 1) & 1, guard, kSiteProducer)) break;
        mbar_arrive_expect_tx(bar_q, kQBytes);
        tma_load_2d(sQ, mq, it.hl * 64, it.row0 + it.qt * 128, bar_q);
        auto put = [&](bool is_v, int blk) {
          const int slot = n % kStrmSlots;
          if (!wait_bounded(ring_empty + slot, ((n / kStrmSlots) & 1) ^ 1u, guard, kSiteProducer)) return false;
          uint8_t* dst = sRing + slot * kStrmSlotBytes;
          mbar_arrive_expect_tx(ring_full + slot, kStrmSlotBytes);
          if (is_v) {
            tma_load_2d(dst, mv, it.row0 + blk * 128, it.hl * 64, ring_full + slot);
            tma_load_2d(dst + kVtChunkBytes, mv, it.row0 + blk * 128 + 64, it.hl * 64, ring_full + slot);
          } else {
            tma_load_2d(dst, mq, kx, it.row0 + blk * 128, ring_full + slot);
          }
          ++n;
          return true;
        };
        ok = put(false, 0);
        for (int j = 1; ok && j < nkv; ++j) ok = put(false, j) && put(true, j - 1);
        if (ok) ok = put(true, nkv - 1);
        ++k;
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // ---------------- products
      const uint64_t dq = smem_desc_sw128(smem_addr(sQ));
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128);
      constexpr uint32_t kIdO = idesc_bf16_f32(128, 64);
      int n = 0;   // ring position of the next operand
      int k = 0;   // items done by this CTA
      int jb = 0;  // blocks done by this CTA (all items): the phase counter of s_read, s_free and o_done
      bool ok = true;
      for (int i = blockIdx.x; ok && i < p.items; i += gridDim.x) {
        Item it;
        if (!decode(i, it)) continue;
        ok = wait_bounded(bar_q, k & 1, guard, kSiteProducer);
        for (int j = 0; ok && j <= nkv; ++j) {
          if (j < nkv) {
            // S_j overwrites the previous block's S once every softmax warp
            // holds its columns, so this product overlaps that softmax.
            const int slot = n % kStrmSlots;
            ok = wait_bounded(ring_full + slot, (n / kStrmSlots) & 1, guard, kSiteMmaFull);
            if (ok && jb + j > 0) ok = wait_bounded(s_read, (jb + j - 1) & 1, guard, kSiteMmaAcc);
            if (!ok) break;
            ++n;
            tc_fence_after_sync();
            const uint64_t dk = smem_desc_sw128(smem_addr(sRing + slot * kStrmSlotBytes));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) tc_mma_bf16(tS, dq + 2 * kk, dk + 2 * kk, kIdS, kk > 0 ? 1u : 0u);
            tc_commit(s_full);
            tc_commit(ring_empty + slot);
            if (j == nkv - 1) tc_commit(q_free);  // the next item's Q may land once this product is done
          }
          if (j > 0) {  // O (+)= P_{j-1} V_{j-1}, once P_{j-1} is written and O rescaled
            const int b = jb + j - 1;  // the block's index among the CTA's blocks
            const int slot = n % kStrmSlots;
            ok = wait_bounded(ring_full + slot, (n / kStrmSlots) & 1, guard, kSiteMmaFull) &&
                 wait_bounded(s_free + (b & 1), (b >> 1) & 1, guard, kSiteMmaAcc);
            // The item's first product overwrites O: the previous item's
            // merge must hold its O in registers.
            if (ok && j == 1 && k > 0) ok = wait_bounded(o_read, (k - 1) & 1, guard, kSiteMmaAcc);
            if (!ok) break;
            ++n;
            tc_fence_after_sync();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const uint64_t dp = smem_desc_sw128(smem_addr(sP + (b & 1) * kStrmPBufBytes + c * kPChunkBytes));
              const uint64_t dv = smem_desc_sw128(smem_addr(sRing + slot * kStrmSlotBytes + c * kVtChunkBytes));
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                tc_mma_bf16(tO + 64u * c, dp + 2 * kk, dv + 2 * kk, kIdO, (j > 1 || kk > 0) ? 1u : 0u);
            }
            tc_commit(o_done + (b & 1));
            tc_commit(ring_empty + slot);
          }
        }
        jb += nkv;
        ++k;
      }
    }
  } else {
    // ---------------- softmax warps
    // Warp (quarter, half) owns query rows 32*quarter.. and the 64 keys of
    // its half of every block, with a running maximum, a row sum and an
    // output accumulator O_half of its own, so the two warps of a row never
    // wait for each other inside the loop; their partial results are merged
    // once at the end of the item.
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tOh = tO + lane_off + 64u * half;  // this warp's rows of O_half
    bool ok = true;
    int k = 0;   // items done by this CTA
    int jb = 0;  // blocks done by this CTA
    for (int i = blockIdx.x; ok && i < p.items; i += gridDim.x) {
      Item it;
      if (!decode(i, it)) continue;
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nkv; ++j) {
        const int b = jb + j;  // the block's index among the CTA's blocks
        ok = __all_sync(0xffffffffu, ok && wait_bounded(s_full, b & 1, guard, kSiteMmaFull));
        if (!ok) break;
        tc_fence_after_sync();
        float v[64];
        {
          uint32_t r0[32], r1[32];
          tmem_ld_32cols_async(tS + lane_off + half * 64, r0);
          tmem_ld_32cols_async(tS + lane_off + half * 64 + 32, r1);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            v[q] = __uint_as_float(r0[q]);
            v[32 + q] = __uint_as_float(r1[q]);
          }
        }
        tc_fence_before_sync();  // S may be overwritten by the next block's product now
        __syncwarp();
        if (lane == 0) mbar_arrive(s_read);
        const int kbase = j * 128 + half * 64;  // key of column 0 of this half
        const bool full = kbase + 64 <= p.seq;
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (full) {  // every column a key of the sequence: two values per max
#pragma unroll
          for (int q = 0; q < 64; q += 2) m4[(q >> 1) & 3] = fmax3(m4[(q >> 1) & 3], v[q], v[q + 1]);
        } else {
#pragma unroll
          for (int q = 0; q < 64; ++q)
            if (kbase + q < p.seq) m4[q & 3] = fmaxf(m4[q & 3], v[q]);
        }
        const float m_blk = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        // The running maximum moves only when the block's exceeds it by more
        // than 8 in log2 units: until then the weights stay <= 2^8 (well inside
        // fp32 and bf16 range) and O needs no rescale; the final division by l
        // is the same either way. A half without keys so far keeps -inf and
        // weight 0 (alpha 1, nothing to rescale).
        const float m_new = (m_blk - m_run) * p.scale_log2 > 8.0f ? m_blk : m_run;  // m_blk on its first keys
        const float alpha = m_new == -INFINITY ? 1.0f : ex2_approx((m_run - m_new) * p.scale_log2);
        const float mb = m_new * p.scale_log2;
        uint32_t w[32];
        float s2[2] = {0.f, 0.f};
        if (full) {
          // Exponent arguments and the row sum on packed fp32 pairs (half the
          // FMA-pipe instructions); the two lanes of a pair are the even and
          // odd columns, so the sums are the same two partial sums as below.
          const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), nmb2 = f2_pack(-mb, -mb);
          uint64_t acc2 = f2_pack(0.f, 0.f);
#pragma unroll
          for (int q = 0; q < 64; q += 2) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(v[q], v[q + 1]), sc2, nmb2), x0, x1);
            const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
            acc2 = f2_add(acc2, f2_pack(e0, e1));
            w[q / 2] = pack2_bf16(e0, e1);
          }
          f2_unpack(acc2, s2[0], s2[1]);
        } else {
#pragma unroll
          for (int q = 0; q < 64; q += 2) {
            const float e0 = kbase + q < p.seq ? ex2_approx(fmaf(v[q], p.scale_log2, -mb)) : 0.f;
            const float e1 = kbase + q + 1 < p.seq ? ex2_approx(fmaf(v[q + 1], p.scale_log2, -mb)) : 0.f;
            s2[0] += e0;
            s2[1] += e1;
            w[q / 2] = pack2_bf16(e0, e1);
          }
        }
        l_run = l_run * alpha + (s2[0] + s2[1]);
        if (b > 1) {  // P buffer b % 2 was last read by the product of block b - 2
          ok = __all_sync(0xffffffffu, wait_bounded(o_done + (b & 1), ((b >> 1) - 1) & 1, guard, kSiteMmaAcc));
          if (!ok) break;
        }
        uint8_t* prow = sP + (b & 1) * kStrmPBufBytes + half * kPChunkBytes + row * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(prow + ((u ^ (row & 7)) << 4)) =
              make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {  // rescale this warp's rows of O_half
          // once the previous block's product has finished writing O
          ok = __all_sync(0xffffffffu,
                          wait_bounded(o_done + ((b - 1) & 1), ((b - 1) >> 1) & 1, guard, kSiteMmaAcc));
          if (!ok) break;
          tc_fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < 64; c += 32) {
            float o[32];
            tmem_ld_32cols(tOh + c, o);
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] *= alpha;
            tmem_st_32cols(tOh + c, o);
          }
        }
        m_run = m_new;
        fence_proxy_async_smem();  // P, written by threads, is read by the tensor cores
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free + (b & 1));
      }
      if (!ok) break;
      // ---- merge the halves: O = (f_0 O_0 + f_1 O_1) / (f_0 l_0 + f_1 l_1), f_h = 2^((m_h - m) s), m = max m_h.
      // The halves' maxima and sums meet in the P buffer of the item's last
      // block: its product is done, and it is next written two blocks on,
      // after every warp has passed this merge.
      const int bl = jb + nkv - 1;
      float* red_max = reinterpret_cast<float*>(sP + (bl & 1) * kStrmPBufBytes);  // [2][128]
      float* red_sum = red_max + 256;                                            // [2][128]
      ok = __all_sync(0xffffffffu, wait_bounded(o_done + (bl & 1), (bl >> 1) & 1, guard, kSiteEpilogue));
      if (ok) {
        red_max[half * 128 + row] = m_run;
        red_sum[half * 128 + row] = l_run;
        __syncwarp();
        if (lane == 0) mbar_arrive(x_bar);
        ok = __all_sync(0xffffffffu, wait_bounded(x_bar, k & 1, guard, kSiteEpilogue));
      }
      if (!ok) break;
      tc_fence_after_sync();
      float o0[32], o1[32];
      tmem_ld_32cols(tO + lane_off + half * 32, o0);       // O_0, this warp's 32 output columns
      tmem_ld_32cols(tO + lane_off + 64 + half * 32, o1);  // O_1, the same columns
      tc_fence_before_sync();  // O may be overwritten by the next item's first product now
      __syncwarp();
      if (lane == 0) mbar_arrive(o_read);
      const int qi = it.qt * 128 + row;
      if (qi < p.seq) {
        const float m0 = red_max[row], m1 = red_max[128 + row];
        const float m = fmaxf(m0, m1);  // finite: key 0 lies in half 0 of block 0
        const float f0 = ex2_approx((m0 - m) * p.scale_log2);
        const float f1 = m1 == -INFINITY ? 0.0f : ex2_approx((m1 - m) * p.scale_log2);
        const float inv = 1.0f / (f0 * red_sum[row] + f1 * red_sum[128 + row]);
        const float g0 = f0 * inv, g1 = f1 * inv;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out[it.shard]) +
                             (static_cast<int64_t>(it.row0) + qi) * p.Dn + it.hl * 64 + half * 32;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = fmaf(o0[8 * u + e], g0, o1[8 * u + e] * g1);
          reinterpret_cast<uint4*>(dst)[u] =
              make_uint4(pack2_bf16(y[0], y[1]), pack2_bf16(y[2], y[3]), pack2_bf16(y[4], y[5]), pack2_bf16(y[6], y[7]));
        }
      }
      jb += nkv;
      ++k;
    }
  }

  // ---- clean-up: after an abort, copies and products in flight finish first
  __syncthreads();
  if (*abort_flag && tid == kStrmSoftmaxWarps * 32) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) {
    }
    tc_commit(drain);
    wait_drain(drain, 0, p.wait_ns);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kStrmSoftmaxWarps) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kCols);
  }
}

// ------------------------------------------------------------------ fp32 (CUDA cores)

template <int DHMAX>
__global__ void __launch_bounds__(kF32Threads) attn_f32_kernel(const float* __restrict__ qkv, int64_t ld_qkv,
                                                                int64_t shard_stride_qkv, float* __restrict__ out,
                                                                int64_t shard_stride_out, int seq, int Dn, int dh,
                                                                int local_heads, float scale) {
  extern __shared__ float smem_f[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* sc = smem_f + warp * seq;  // this warp's score row
  const int gh = blockIdx.y, b = blockIdx.z;
  const int shard = gh / local_heads, hl = gh % local_heads;
  const int qi = blockIdx.x * (kF32Threads / 32) + warp;
  if (qi >= seq) return;
  const float* base = qkv + shard * shard_stride_qkv;
  const int64_t row0 = int64_t(b) * seq;
  const float* q = base + (row0 + qi) * ld_qkv + hl * dh;
  float qr[DHMAX / 32];
#pragma unroll
  for (int u = 0; u < DHMAX / 32; ++u) qr[u] = (u * 32 + lane < dh) ? q[u * 32 + lane] : 0.f;
  float mx = -INFINITY;
  for (int j = 0; j < seq; ++j) {
    const float* k = base + (row0 + j) * ld_qkv + Dn + hl * dh;
    float part = 0.f;
#pragma unroll
    for (int u = 0; u < DHMAX / 32; ++u)
      if (u * 32 + lane < dh) part += qr[u] * k[u * 32 + lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    const float s = part * scale;
    if (lane == 0) sc[j] = s;
    mx = fmaxf(mx, s);
  }
  __syncwarp();
  float sum = 0.f;
  for (int j = lane; j < seq; j += 32) {
    const float e = expf(sc[j] - mx);
    sc[j] = e;
    sum += e;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  __syncwarp();
  float acc[DHMAX / 32];
#pragma unroll
  for (int u = 0; u < DHMAX / 32; ++u) acc[u] = 0.f;
  for (int j = 0; j < seq; ++j) {
    const float* v = base + (row0 + j) * ld_qkv + 2 * Dn + hl * dh;
    const float pj = sc[j];
#pragma unroll
    for (int u = 0; u < DHMAX / 32; ++u)
      if (u * 32 + lane < dh) acc[u] += pj * v[u * 32 + lane];
  }
  float* o = out + shard * shard_stride_out + (row0 + qi) * Dn + hl * dh;
#pragma unroll
  for (int u = 0; u < DHMAX / 32; ++u)
    if (u * 32 + lane < dh) o[u * 32 + lane] = acc[u] / sum;
}

}  // namespace

// The streaming kernel by default (any length; as fast as the exact one up to
// 512 tokens); TPMLP_ATTN_KERNEL=0 selects the exact kernel where it applies
// (seq <= 512). Read at every launch, so a process can compare the two.
int attn_kernel_choice(int seq) {
  if (seq > 512) return 1;
  const char* v = getenv("TPMLP_ATTN_KERNEL");
  return (v && atoi(v) == 0) ? 0 : 1;
}

cudaError_t launch_attention_tc(const AttnLaunch& a, cudaStream_t s) {
  if (a.batch <= 0 || a.seq <= 0) return cudaSuccess;
  if (a.seq % 8 != 0 || a.n < 1 || a.n > kMaxGroups) return cudaErrorInvalidValue;
  AttnParams p;
  memset(&p, 0, sizeof(p));
  for (int i = 0; i < a.n; ++i) {
    p.map_qkv[i] = *a.map_qkv[i];
    p.map_vt[i] = *a.map_vt[i];
    p.out[i] = a.out[i];
  }
  p.seq = a.seq;
  p.Dn = a.Dn;
  p.local_heads = a.local_heads;
  p.scale_log2 = 1.4426950408889634f / sqrtf(64.0f);
  p.wait_ns = a.wait_ns;
  p.status = a.status;
  dim3 grid(static_cast<unsigned>((a.seq + 127) / 128), static_cast<unsigned>(a.n * a.local_heads),
            static_cast<unsigned>(a.batch));
  if (attn_kernel_choice(a.seq) == 1) {
    cudaError_t e = cudaFuncSetAttribute(attn_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kStrmSmem));
    if (e != cudaSuccess) return e;
    // Work items (query tile, head, sequence) taken by a persistent grid of
    // the CTAs that fit at once (two per SM), each running its items through
    // one pipeline; TPMLP_ATTN_PERSIST=0 (read at every launch) launches one
    // CTA per item instead.
    p.q_tiles = static_cast<int>(grid.x);
    p.heads = static_cast<int>(grid.y);
    p.items = static_cast<int>(grid.x * grid.y * grid.z);
    // Two CTAs per SM by design (launch bounds, 112 KB of shared memory and
    // 256 TMEM columns each); the occupancy calculator reports one here, so
    // the grid is sized from the design. CTAs share nothing, so a grid that
    // did not fit at once would only run in two waves.
    int ctas = p.items;
    const char* pv = getenv("TPMLP_ATTN_PERSIST");
    if (!(pv && *pv && atoi(pv) == 0) && int64_t(2) * num_sms() < ctas) ctas = 2 * num_sms();
    return launch_pdl(attn_stream_kernel, dim3(static_cast<unsigned>(ctas)), dim3(kStrmThreads), kStrmSmem, s, p);
  }
  const int nkv = (a.seq + 127) / 128, nch = (a.seq + 63) / 64;
  const uint32_t smem = attn_smem_bytes(nkv, nch);
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(attn_smem_bytes(4, 8)));
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_tc_kernel, grid, dim3(kAttnThreads), smem, s, p);
}

cudaError_t launch_attention_f32(const float* qkv, int64_t T, int n, int Dn, int dh, int local_heads, int batch,
                                 int seq, float* out, cudaStream_t s) {
  if (batch <= 0 || seq <= 0) return cudaSuccess;
  if (dh > 128 || seq > 8192) return cudaErrorInvalidValue;
  const size_t smem = size_t(kF32Threads / 32) * seq * sizeof(float);
  for (auto k : {attn_f32_kernel<32>, attn_f32_kernel<64>, attn_f32_kernel<128>}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 4 * 8192 * 4);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(static_cast<unsigned>((seq + 3) / 4), static_cast<unsigned>(n * local_heads), static_cast<unsigned>(batch));
  const float scale = 1.0f / sqrtf(static_cast<float>(dh));
  const int64_t ld = 3 * int64_t(Dn);
  if (dh <= 32)
    attn_f32_kernel<32><<<grid, kF32Threads, smem, s>>>(qkv, ld, T * ld, out, T * Dn, seq, Dn, dh, local_heads, scale);
  else if (dh <= 64)
    attn_f32_kernel<64><<<grid, kF32Threads, smem, s>>>(qkv, ld, T * ld, out, T * Dn, seq, Dn, dh, local_heads, scale);
  else
    attn_f32_kernel<128><<<grid, kF32Threads, smem, s>>>(qkv, ld, T * ld, out, T * Dn, seq, Dn, dh, local_heads,
                                                          scale);
  return cudaGetLastError();
}

}  // namespace tpmlp
