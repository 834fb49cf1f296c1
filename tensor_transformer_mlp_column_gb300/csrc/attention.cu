// attention.cu — the local attention of head-split tensor parallelism
// (duoan.github.io "Tensor Parallelism in Megatron-LM", §4): for every
// sequence b and head h of every rank, O = softmax(Q K^T / sqrt(d_h)) V with
// no mask, reading Q, K from the rank's QKV projection [T, 3 D/n] and V from
// its transpose V^T [D/n, T], and writing O into the rank's [T, D/n] block.
//
// Tensor-core kernel (bf16, d_h = 64, seq <= 512, seq % 8 == 0): one CTA of
// four warps per (128-query tile, head, sequence).
//   thread 0 : TMA-loads the Q tile, all keys and all of V^T for the head
//              into 128-byte-swizzled shared memory (one mbarrier), then
//              issues S = Q K^T (M=128, N=128 per key block, K=16 steps)
//              into tensor memory: the whole score row, up to 512 columns
//   all 128  : thread r owns query row r (TMEM lane r): one pass over its
//              scores for the row maximum, a second for p = 2^((s - max) *
//              log2(e) / sqrt(d_h)) and their fp32 sum, writing p as bf16
//              into shared memory in the 128-byte-swizzled K-major layout of
//              an MMA operand; then O (+)= P V^T-chunk (M=128, N=64) into
//              TMEM columns 0..63, in phases of 256 keys (P buffer of
//              64 KB); finally O / sum rounded to bf16.
// The softmax is exact (the full row is in tensor memory), not the running
// rescale of a streaming kernel. Every wait is bounded; on a timeout the CTA
// records the site, drains its copies and MMAs and frees its tensor memory.
//
// fp32 kernel (any d_h <= 128, seq <= 512): one warp per query row, scores
// in shared memory, the same two passes, on the CUDA cores.
#include "device.cuh"
#include "internal.h"

namespace tpmlp {

namespace {

constexpr int kAttnThreads = 128;
constexpr uint32_t kQBytes = 128 * 128;       // 128 query rows x 64 bf16
constexpr uint32_t kKBlockBytes = 128 * 128;  // 128 key rows x 64 bf16
constexpr uint32_t kVtChunkBytes = 64 * 128;  // 64 d-rows x 64 keys
constexpr uint32_t kPChunkBytes = 128 * 128;  // 128 query rows x 64 keys
constexpr int kPhaseChunks = 4;               // P chunks per phase (256 keys)

struct AttnParams {
  CUtensorMap map_qkv[kMaxGroups];  // QKV_i [T, 3 Dn] bf16, boxes 64 x 128
  CUtensorMap map_vt[kMaxGroups];   // V_i^T [Dn, T] bf16 (row pitch T8), boxes 64 x 64
  void* out[kMaxGroups];            // O_i [T, Dn]
  int seq, Dn, local_heads;
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
         uint32_t(nch < kPhaseChunks ? nch : kPhaseChunks) * kPChunkBytes + 64;
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
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + (nch < kPhaseChunks ? nch : kPhaseChunks) * kPChunkBytes);
  uint64_t* bar_load = bars;
  uint64_t* bar_mma = bars + 1;
  uint64_t* bar_drain = bars + 2;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 3);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4);

  const int qt = blockIdx.x, gh = blockIdx.y, b = blockIdx.z;
  const int shard = gh / p.local_heads, hl = gh % p.local_heads;
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t tmem_cols = nkv <= 1 ? 128u : (nkv <= 2 ? 256u : 512u);

  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, tmem_cols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const WaitGuard guard{abort_flag, p.wait_ns, p.status};

  const int32_t row0 = b * p.seq;  // first token of the sequence
  if (tid == 0) {
    const CUtensorMap* mq = &p.map_qkv[shard];
    const CUtensorMap* mv = &p.map_vt[shard];
    mbar_arrive_expect_tx(bar_load, kQBytes + nkv * kKBlockBytes + nch * kVtChunkBytes);
    tma_load_2d(sQ, mq, hl * 64, row0 + qt * 128, bar_load);
    for (int j = 0; j < nkv; ++j) tma_load_2d(sK + j * kKBlockBytes, mq, p.Dn + hl * 64, row0 + j * 128, bar_load);
    for (int c = 0; c < nch; ++c) tma_load_2d(sVt + c * kVtChunkBytes, mv, row0 + c * 64, hl * 64, bar_load);
  }
  bool ok = wait_bounded(bar_load, 0, guard, kSiteProducer);
  uint32_t mma_phase = 0;
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
  ok = ok && wait_bounded(bar_mma, mma_phase, guard, kSiteMmaFull);
  mma_phase ^= 1u;

  // ---- softmax: thread tid owns query row tid (TMEM lane tid)
  tc_fence_after_sync();
  const uint32_t t_row = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  float mx = -INFINITY;
  if (ok) {
    for (int g = 0; g < nkv * 4; ++g) {
      float v[32];
      tmem_ld_32cols(t_row + g * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (g * 32 + j < p.seq) mx = fmaxf(mx, v[j]);
    }
  }
  const float mb = mx * p.scale_log2;
  float sum = 0.f;
  for (int ph = 0; ph * kPhaseChunks < nch; ++ph) {
    if (ph > 0) {  // the previous phase's products must have read P before it is overwritten
      ok = ok && wait_bounded(bar_mma, mma_phase, guard, kSiteMmaAcc);
      mma_phase ^= 1u;
    }
    const int c0 = ph * kPhaseChunks;
    const int c1 = (c0 + kPhaseChunks < nch) ? c0 + kPhaseChunks : nch;
    if (ok) {
      for (int c = c0; c < c1; ++c) {
        uint8_t* prow = sP + (c - c0) * kPChunkBytes + tid * 128;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
          tmem_ld_32cols(t_row + c * 64 + half * 32, v);
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const int col = c * 64 + half * 32 + j;
            const float e0 = col < p.seq ? exp2f(fmaf(v[j], p.scale_log2, -mb)) : 0.f;
            const float e1 = col + 1 < p.seq ? exp2f(fmaf(v[j + 1], p.scale_log2, -mb)) : 0.f;
            sum += e0 + e1;
            w[j / 2] = pack2_bf16(e0, e1);
          }
          // 16-byte unit u of a 128-byte row r sits at unit u ^ (r % 8).
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(prow + ((((half * 4 + q) ^ (tid & 7))) << 4)) =
                make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
    }
    fence_proxy_async_smem();  // P, written by threads, is read by the tensor cores
    tc_fence_before_sync();
    __syncthreads();
    if (tid == 0 && ok && !*abort_flag) {
      tc_fence_after_sync();
      constexpr uint32_t kIdO = idesc_bf16_f32(128, 64);
      for (int c = c0; c < c1; ++c) {
        const uint64_t dp = smem_desc_sw128(smem_addr(sP + (c - c0) * kPChunkBytes));
        const uint64_t dv = smem_desc_sw128(smem_addr(sVt + c * kVtChunkBytes));
#pragma unroll
        for (int k = 0; k < 4; ++k) tc_mma_bf16(tmem, dp + 2 * k, dv + 2 * k, kIdO, (c > 0 || k > 0) ? 1u : 0u);
      }
      tc_commit(bar_mma);
    }
  }
  ok = ok && !*abort_flag && wait_bounded(bar_mma, mma_phase, guard, kSiteEpilogue);

  // ---- O / sum -> bf16
  if (ok) {
    tc_fence_after_sync();
    float o0[32], o1[32];
    tmem_ld_32cols(t_row, o0);
    tmem_ld_32cols(t_row + 32, o1);
    const int qi = qt * 128 + tid;
    if (qi < p.seq) {
      const float inv = 1.0f / sum;
      __nv_bfloat16* dst =
          static_cast<__nv_bfloat16*>(p.out[shard]) + (static_cast<int64_t>(row0) + qi) * p.Dn + hl * 64;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        reinterpret_cast<uint4*>(dst)[u] =
            make_uint4(pack2_bf16(o0[8 * u] * inv, o0[8 * u + 1] * inv), pack2_bf16(o0[8 * u + 2] * inv, o0[8 * u + 3] * inv),
                       pack2_bf16(o0[8 * u + 4] * inv, o0[8 * u + 5] * inv), pack2_bf16(o0[8 * u + 6] * inv, o0[8 * u + 7] * inv));
#pragma unroll
      for (int u = 0; u < 4; ++u)
        reinterpret_cast<uint4*>(dst)[4 + u] =
            make_uint4(pack2_bf16(o1[8 * u] * inv, o1[8 * u + 1] * inv), pack2_bf16(o1[8 * u + 2] * inv, o1[8 * u + 3] * inv),
                       pack2_bf16(o1[8 * u + 4] * inv, o1[8 * u + 5] * inv), pack2_bf16(o1[8 * u + 6] * inv, o1[8 * u + 7] * inv));
    }
  }

  // ---- clean-up: after an abort, let copies and products in flight finish first
  __syncthreads();
  if (*abort_flag && tid == 0) {
    wait_drain(bar_load, 0, p.wait_ns);
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

// ------------------------------------------------------------------ fp32 (CUDA cores)

template <int DHMAX>
__global__ void __launch_bounds__(kAttnThreads) attn_f32_kernel(const float* __restrict__ qkv, int64_t ld_qkv,
                                                                int64_t shard_stride_qkv, float* __restrict__ out,
                                                                int64_t shard_stride_out, int seq, int Dn, int dh,
                                                                int local_heads, float scale) {
  extern __shared__ float smem_f[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* sc = smem_f + warp * seq;  // this warp's score row
  const int gh = blockIdx.y, b = blockIdx.z;
  const int shard = gh / local_heads, hl = gh % local_heads;
  const int qi = blockIdx.x * (kAttnThreads / 32) + warp;
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

cudaError_t launch_attention_tc(const AttnLaunch& a, cudaStream_t s) {
  if (a.batch <= 0 || a.seq <= 0) return cudaSuccess;
  if (a.seq > 512 || a.seq % 8 != 0 || a.n < 1 || a.n > kMaxGroups) return cudaErrorInvalidValue;
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
  const int nkv = (a.seq + 127) / 128, nch = (a.seq + 63) / 64;
  const uint32_t smem = attn_smem_bytes(nkv, nch);
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(attn_smem_bytes(4, 8)));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((a.seq + 127) / 128), static_cast<unsigned>(a.n * a.local_heads),
            static_cast<unsigned>(a.batch));
  attn_tc_kernel<<<grid, kAttnThreads, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attention_f32(const float* qkv, int64_t T, int n, int Dn, int dh, int local_heads, int batch,
                                 int seq, float* out, cudaStream_t s) {
  if (batch <= 0 || seq <= 0) return cudaSuccess;
  if (dh > 128 || seq > 512) return cudaErrorInvalidValue;
  const size_t smem = size_t(kAttnThreads / 32) * seq * sizeof(float);
  dim3 grid(static_cast<unsigned>((seq + 3) / 4), static_cast<unsigned>(n * local_heads), static_cast<unsigned>(batch));
  const float scale = 1.0f / sqrtf(static_cast<float>(dh));
  const int64_t ld = 3 * int64_t(Dn);
  if (dh <= 32)
    attn_f32_kernel<32><<<grid, kAttnThreads, smem, s>>>(qkv, ld, T * ld, out, T * Dn, seq, Dn, dh, local_heads, scale);
  else if (dh <= 64)
    attn_f32_kernel<64><<<grid, kAttnThreads, smem, s>>>(qkv, ld, T * ld, out, T * Dn, seq, Dn, dh, local_heads, scale);
  else
    attn_f32_kernel<128><<<grid, kAttnThreads, smem, s>>>(qkv, ld, T * ld, out, T * Dn, seq, Dn, dh, local_heads,
                                                          scale);
  return cudaGetLastError();
}

}  // namespace tpmlp
