// block.cu — the row-wise kernels of the FFN half of a transformer block
// (ai-hpc.org "LLM Lab Notes 06", §2 steps 5-8): the layer norm in front of
// the first product, and in the backward pass the gradient through that
// norm, fused with the shard-ordered sum of the input-gradient partials and
// the residual's pass-through gradient.
//
// Both kernels give one CTA of 256 threads to one token row at a time
// (persistent over rows). The row is staged in shared memory as fp32, so the
// HBM traffic is one read of every input row and one write of every output
// row; the statistics are exact two-pass fp32 (mean first, then the mean of
// squared deviations), summed in a fixed order, so results are reproducible.
#include "device.cuh"
#include "internal.h"

namespace tpmlp {

namespace {

constexpr int kRowThreads = 256;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over the CTA; every thread gets the result. `red` holds 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();  // the previous call's readers are done with `red`
  if (l == 0) red[w] = v;
  __syncthreads();
  return warp_sum(l < (kRowThreads >> 5) ? red[l] : 0.f);
}

// 8 consecutive elements <-> 8 floats (16 bytes of bf16, 32 bytes of fp32).
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&f)[8]) {
  uint4 w = __ldcs(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 t = __bfloat1622float2(h[j]);
    f[2 * j] = t.x;
    f[2 * j + 1] = t.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float (&f)[8]) {
  const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
  const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
  f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w, f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&f)[8]) {
  uint4 w;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
  for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
  *reinterpret_cast<uint4*>(p) = w;
}
__device__ __forceinline__ void store8(float* p, const float (&f)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void from_f(float& d, float v) { d = v; }
__device__ __forceinline__ void from_f(__nv_bfloat16& d, float v) { d = __float2bfloat16_rn(v); }

// Stage row `src` (D elements of E) into xs as fp32 and return this thread's
// share of its sum. vec: D % 8 == 0, so the row splits into 8-element chunks.
template <typename E>
__device__ __forceinline__ float stage_row(const E* __restrict__ src, int D, bool vec, float* xs) {
  float s = 0.f;
  if (vec) {
    for (int c = threadIdx.x; c < D / 8; c += kRowThreads) {
      float f[8];
      load8(src + 8 * c, f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        xs[8 * c + j] = f[j];
        s += f[j];
      }
    }
  } else {
    for (int j = threadIdx.x; j < D; j += kRowThreads) {
      const float f = to_f(src[j]);
      xs[j] = f;
      s += f;
    }
  }
  return s;
}

// mean and r = 1 / sqrt(var + eps) of the staged row (two passes over xs).
__device__ __forceinline__ void row_stats(const float* xs, float sum_part, int D, float eps, float* red, float& mean,
                                          float& r) {
  mean = block_sum(sum_part, red) / static_cast<float>(D);
  float q = 0.f;
  for (int j = threadIdx.x; j < D; j += kRowThreads) {
    const float d = xs[j] - mean;
    q += d * d;
  }
  const float var = block_sum(q, red) / static_cast<float>(D);
  r = 1.0f / sqrtf(var + eps);
}

// y = (x - mean(x)) / sqrt(var(x) + eps) per row, var the biased variance;
// no scale or shift parameters.
template <typename E>
__global__ void __launch_bounds__(kRowThreads) layer_norm_kernel(const E* __restrict__ x, int64_t T, int D, float eps,
                                                                 E* __restrict__ y) {
  extern __shared__ float smem_ln[];
  float* red = smem_ln;       // 32
  float* xs = smem_ln + 32;   // D
  const bool vec = (D % 8) == 0;
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    const E* xr = x + t * D;
    E* yr = y + t * D;
    const float s = stage_row(xr, D, vec, xs);  // each thread reads back only what it staged until the barrier
    float mean, r;
    row_stats(xs, s, D, eps, red, mean, r);
    if (vec) {
      for (int c = threadIdx.x; c < D / 8; c += kRowThreads) {
        float f[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = (xs[8 * c + j] - mean) * r;
        store8(yr + 8 * c, f);
      }
    } else {
      for (int j = threadIdx.x; j < D; j += kRowThreads) from_f(yr[j], (xs[j] - mean) * r);
    }
    __syncthreads();  // xs is refilled for the next row
  }
}

// dx = dout + r (g - mean(g) - y mean(g y)) per row, with y the row's
// normalised input, r its 1/sqrt(var + eps), and g = ((G_0 + G_1) + ...) +
// G_{n-1} the shard-ordered sum of the n input-gradient partials ([n][T][D]
// fp32; n = 1 when the sum was already taken).
template <typename E>
__global__ void __launch_bounds__(kRowThreads) layer_norm_bwd_kernel(const float* __restrict__ G, int n,
                                                                     const E* __restrict__ x,
                                                                     const E* __restrict__ dout, int64_t T, int D,
                                                                     float eps, float* __restrict__ dx) {
  extern __shared__ float smem_lnb[];
  float* red = smem_lnb;           // 32
  float* xs = smem_lnb + 32;       // D: x, then y
  float* gs = smem_lnb + 32 + D;   // D: g
  const bool vec = (D % 8) == 0;
  const int64_t gstride = T * D;
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    const int64_t row = t * D;
    const float s = stage_row(x + row, D, vec, xs);
    // g: the n partials of each chunk are loaded before they are added.
    if (vec) {
      for (int c = threadIdx.x; c < D / 8; c += kRowThreads) {
        float acc[8];
        load8(G + row + 8 * c, acc);
        for (int k = 1; k < n; ++k) {
          float f[8];
          load8(G + k * gstride + row + 8 * c, f);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] += f[j];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) gs[8 * c + j] = acc[j];
      }
    } else {
      for (int j = threadIdx.x; j < D; j += kRowThreads) {
        float acc = G[row + j];
        for (int k = 1; k < n; ++k) acc += G[k * gstride + row + j];
        gs[j] = acc;
      }
    }
    float mean, r;
    row_stats(xs, s, D, eps, red, mean, r);  // its barriers also publish gs
    float sg = 0.f, sgy = 0.f;
    for (int j = threadIdx.x; j < D; j += kRowThreads) {
      const float yv = (xs[j] - mean) * r;
      xs[j] = yv;
      sg += gs[j];
      sgy += gs[j] * yv;
    }
    const float mg = block_sum(sg, red) / static_cast<float>(D);
    const float mgy = block_sum(sgy, red) / static_cast<float>(D);
    if (vec) {
      for (int c = threadIdx.x; c < D / 8; c += kRowThreads) {
        float d[8], f[8];
        load8(dout + row + 8 * c, d);
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = d[j] + r * (gs[8 * c + j] - mg - xs[8 * c + j] * mgy);
        store8(dx + row + 8 * c, f);
      }
    } else {
      for (int j = threadIdx.x; j < D; j += kRowThreads)
        dx[row + j] = to_f(dout[row + j]) + r * (gs[j] - mg - xs[j] * mgy);
    }
    __syncthreads();
  }
}

// out[j] += res[j] (fp32), for the fp32 path's fused sum.
__global__ void add_residual_f32_kernel(float* __restrict__ out, const float* __restrict__ res, int64_t count) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t j = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; j < count; j += stride) out[j] = out[j] + res[j];
}

template <typename K>
int row_grid(K kern, size_t smem, int64_t T) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRowThreads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int64_t cap = int64_t(num_sms()) * per_sm;
  return static_cast<int>(T < cap ? T : cap);
}

template <typename K>
cudaError_t set_smem(K kern, size_t smem) {
  if (smem <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
}

}  // namespace

size_t layer_norm_max_d() { return (200 * 1024) / 8 - 64; }

cudaError_t launch_layer_norm(const void* x, int64_t T, int D, float eps, int is_bf16, void* y, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const size_t smem = (32 + size_t(D)) * sizeof(float);
  if (is_bf16) {
    auto k = layer_norm_kernel<__nv_bfloat16>;
    cudaError_t e = set_smem(k, smem);
    if (e != cudaSuccess) return e;
    k<<<row_grid(k, smem, T), kRowThreads, smem, s>>>(static_cast<const __nv_bfloat16*>(x), T, D, eps,
                                                     static_cast<__nv_bfloat16*>(y));
  } else {
    auto k = layer_norm_kernel<float>;
    cudaError_t e = set_smem(k, smem);
    if (e != cudaSuccess) return e;
    k<<<row_grid(k, smem, T), kRowThreads, smem, s>>>(static_cast<const float*>(x), T, D, eps,
                                                     static_cast<float*>(y));
  }
  return cudaGetLastError();
}

cudaError_t launch_layer_norm_bwd(const float* G, int n, const void* x, const void* dout, int64_t T, int D, float eps,
                                  int is_bf16, float* dx, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const size_t smem = (32 + 2 * size_t(D)) * sizeof(float);
  if (is_bf16) {
    auto k = layer_norm_bwd_kernel<__nv_bfloat16>;
    cudaError_t e = set_smem(k, smem);
    if (e != cudaSuccess) return e;
    k<<<row_grid(k, smem, T), kRowThreads, smem, s>>>(G, n, static_cast<const __nv_bfloat16*>(x),
                                                     static_cast<const __nv_bfloat16*>(dout), T, D, eps, dx);
  } else {
    auto k = layer_norm_bwd_kernel<float>;
    cudaError_t e = set_smem(k, smem);
    if (e != cudaSuccess) return e;
    k<<<row_grid(k, smem, T), kRowThreads, smem, s>>>(G, n, static_cast<const float*>(x),
                                                     static_cast<const float*>(dout), T, D, eps, dx);
  }
  return cudaGetLastError();
}

cudaError_t launch_add_residual_f32(float* out, const float* res, int64_t count, cudaStream_t s) {
  if (count <= 0) return cudaSuccess;
  const int64_t want = (count + kRowThreads - 1) / kRowThreads;
  const int64_t cap = int64_t(num_sms()) * 8;
  add_residual_f32_kernel<<<static_cast<int>(want < cap ? want : cap), kRowThreads, 0, s>>>(out, res, count);
  return cudaGetLastError();
}

}  // namespace tpmlp
