// gemm_common.cuh — what the tensor-core GEMM kernels share: the launch
// parameter block, the tile order, and the epilogue output treatments.
#pragma once

#include "device.cuh"
#include "internal.h"

namespace tpmlp {

constexpr int BM = 128;  // rows of a tile per CTA
constexpr int BK = 64;   // K per pipeline stage: one 128-byte swizzle row of bf16
constexpr int kThreads = 192;  // warp 0 TMA producer, warp 1 MMA issuer, warps 2..5 epilogue

struct KParams {
  CUtensorMap map_a[kMaxGroups];
  CUtensorMap map_b[kMaxGroups];
  void* out[kMaxGroups];
  void* out2[kMaxGroups];           // kEpiGeluSaveP: fp32 pre-activation; kEpiBwdAct: H (bf16); row pitch ldo
  CUtensorMap map_out[kMaxGroups];  // kEpiF32Tma: fp32 output per group, 32 x 32 boxes, 128-byte swizzle
  const void* aux_p[kMaxGroups];    // kEpiBwdAct: P per group (fp32, row pitch ldo)
  void* aux_ht[kMaxGroups];         // kEpiBf16: V^T per group (bf16, row pitch ldt)
  int64_t ldo, ldt;
  int M, N;
  int groups;
  int chain;
  int m_blocks, n_blocks, k_blocks;  // tile-grid units of the kernel that runs (see decode_tile)
  int tiles;
  uint64_t wait_ns;
  int* status;     // device status word (bounded waits record their site here)
  int inject;      // test hook: > 0 withholds that fill (1-based) in every CTA
  int group_m;     // tile order: bands of group_m tile rows, rows fastest inside a band (1 = columns fastest)
  int shared;      // kSharedNone / kSharedA / kSharedB: an operand that every group reads
  int stream_out;  // 1: epilogue stores bypass L2 retention (evict-first)
  int load_hint;   // pair kernel: L2 policy kinds (l2_policy) of the M x K operand's loads (bits 0-1) and the N x K one's (2-3)
  const __nv_bfloat16* resid;  // kEpiF32 / kEpiF32Tma: residual [M][ldo] added to the accumulator, or null
  int64_t slice_rows;          // kEpiF32, chain: output row m goes to row m % slice_rows of out[m / slice_rows]
  int vt_col0;                 // kEpiBf16 with aux_ht: columns >= vt_col0 go transposed to aux_ht (row pitch ldt)
  int mn_major;                // TcMajor bits: MN-major operands and their map form
};

// Maps a tile index to (group, M block, N block). The tiles form a grid of
// `rows` x `cols`, walked in bands of group_m rows with rows fastest inside a
// band, so the tiles in flight together cover about group_m rows x
// (tiles in flight / group_m) columns and each operand panel is fetched from
// DRAM about once per band instead of once per tile.
//   shared A (every group reads the same M x K operand): rows = M blocks,
//     cols = the groups' N blocks side by side;
//   shared B (every group reads the same N x K operand): rows = the groups'
//     M blocks stacked, cols = N blocks;
//   otherwise each group's grid in turn (chain mode: the one output grid).
// "Blocks" are the kernel's tile units.
struct TileGrid {
  int chain, shared, groups, m_blocks, n_blocks, group_m;
};
__device__ __forceinline__ void decode_tile(const TileGrid& p, int tile, int& g, int& mb, int& nb) {
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
__device__ __forceinline__ void decode_tile(const KParams& p, int tile, int& g, int& mb, int& nb) {
  decode_tile(TileGrid{p.chain, p.shared, p.groups, p.m_blocks, p.n_blocks, p.group_m}, tile, g, mb, nb);
}

// Debug build: a decoded tile must lie inside the launch's tile grid. Every
// role of a kernel checks the same tiles, so all of them skip a bad one alike.
__device__ __forceinline__ bool tile_ok(const TileGrid& p, int* status, int g, int mb, int nb) {
  return TPMLP_DCHECK(g >= 0 && g < p.groups && mb >= 0 && mb < p.m_blocks && nb >= 0 && nb < p.n_blocks, status,
                      kChkTile);
}
__device__ __forceinline__ bool tile_ok(const KParams& p, int g, int mb, int nb) {
  return tile_ok(TileGrid{p.chain, p.shared, p.groups, p.m_blocks, p.n_blocks, p.group_m}, p.status, g, mb, nb);
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
// The bf16 residual of output row m, columns n0..n0+31 (chunks of 8 past N
// stay zero; N is a multiple of 8 on this path). Loaded before the
// accumulator is read so that the load's latency overlaps tcgen05.ld.
__device__ __forceinline__ void load_residual(const KParams& p, int64_t m, int n0, uint4 (&r)[4]) {
  const __nv_bfloat16* src = p.resid + m * p.ldo + n0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    r[j] = (n0 + 8 * j + 8 <= p.N) ? __ldcs(reinterpret_cast<const uint4*>(src + 8 * j)) : make_uint4(0, 0, 0, 0);
}

// v[j] = residual[j] + v[j] (the residual added to the finished sum).
__device__ __forceinline__ void add_residual(const uint4 (&r)[4], float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r[j]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      v[8 * j + 2 * e] = f.x + v[8 * j + 2 * e];
      v[8 * j + 2 * e + 1] = f.y + v[8 * j + 2 * e + 1];
    }
  }
}

template <int EPI>
__device__ __forceinline__ void epilogue_store(const KParams& p, int g, int64_t m, int n0, const float (&v)[32]) {
  if constexpr (EPI == kEpiBf16) {
    // acc rounded to bf16, row-major; with aux_ht, columns from vt_col0 on
    // are written transposed instead (column c - vt_col0 of aux_ht's rows;
    // the 32 lanes hold 32 consecutive rows, so each column is 64 contiguous
    // bytes per warp).
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out[g]) + m * p.ldo + n0;
    __nv_bfloat16* vt = static_cast<__nv_bfloat16*>(p.aux_ht[g]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (vt && n0 + 8 * j >= p.vt_col0 && n0 + 8 * j + 8 <= p.N) {
        __nv_bfloat16* t = vt + int64_t(n0 + 8 * j - p.vt_col0) * p.ldt + m;
#pragma unroll
        for (int e = 0; e < 8; ++e) t[int64_t(e) * p.ldt] = __float2bfloat16_rn(v[8 * j + e]);
      } else if (n0 + 8 * j + 8 <= p.N) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
        w.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
        w.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
        w.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
        store16(out + 8 * j, w, p.stream_out);
      }
    }
  } else if constexpr (EPI == kEpiGeluBf16 || EPI == kEpiGeluSaveP) {
    // H = GeLU(acc), bf16, row-major (and, saving P, acc itself in fp32).
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out[g]) + m * p.ldo + n0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (n0 + 8 * j + 8 <= p.N) {
        uint4 w;
        w.x = pack_bf16x2(gelu_bf16_fast(v[8 * j + 0]), gelu_bf16_fast(v[8 * j + 1]));
        w.y = pack_bf16x2(gelu_bf16_fast(v[8 * j + 2]), gelu_bf16_fast(v[8 * j + 3]));
        w.z = pack_bf16x2(gelu_bf16_fast(v[8 * j + 4]), gelu_bf16_fast(v[8 * j + 5]));
        w.w = pack_bf16x2(gelu_bf16_fast(v[8 * j + 6]), gelu_bf16_fast(v[8 * j + 7]));
        store16(out + 8 * j, w, p.stream_out);
        if constexpr (EPI == kEpiGeluSaveP) {
          float* P = static_cast<float*>(p.out2[g]) + m * p.ldo + n0 + 8 * j;
          store16(P, make_uint4(__float_as_uint(v[8 * j]), __float_as_uint(v[8 * j + 1]), __float_as_uint(v[8 * j + 2]),
                                __float_as_uint(v[8 * j + 3])), false);
          store16(P + 4, make_uint4(__float_as_uint(v[8 * j + 4]), __float_as_uint(v[8 * j + 5]),
                                    __float_as_uint(v[8 * j + 6]), __float_as_uint(v[8 * j + 7])), false);
        }
      }
    }
  } else if constexpr (EPI == kEpiF32) {
    // With slice_rows, the rows are cut into rank slices, each its own buffer
    // (the scattered output of a sequence-parallel sum; chain mode, g = 0).
    float* out = p.slice_rows ? static_cast<float*>(p.out[m / p.slice_rows]) + (m % p.slice_rows) * p.ldo + n0
                              : static_cast<float*>(p.out[g]) + m * p.ldo + n0;
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
    // With P from aux_p: dP = dH * GeLU'(P) to out and H = GeLU(P) to out2,
    // both bf16 row-major [T][ldo].
    const float* P = static_cast<const float*>(p.aux_p[g]) + m * p.ldo + n0;
    __nv_bfloat16* dP = static_cast<__nv_bfloat16*>(p.out[g]) + m * p.ldo + n0;
    __nv_bfloat16* H = static_cast<__nv_bfloat16*>(p.out2[g]) + m * p.ldo + n0;
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
      w.x = pack_bf16x2(h[0], h[1]);
      w.y = pack_bf16x2(h[2], h[3]);
      w.z = pack_bf16x2(h[4], h[5]);
      w.w = pack_bf16x2(h[6], h[7]);
      store16(H + 8 * j, w, false);
    }
  }
}

// Launches the CTA-pair kernel with epilogue `epi`; kp's tile units must
// match (256-row M blocks, 256-column N blocks).
cudaError_t launch_pair(const KParams& kp, int epi, cudaStream_t s);

}  // namespace tpmlp
