// block.cu — the row-wise kernels of the FFN half of a transformer block
// (ai-hpc.org "LLM Lab Notes 06", §2 steps 5-8): the layer norm in front of
// the first product, and in the backward pass the gradient through that
// norm, fused with the shard-ordered sum of the input-gradient partials and
// the residual's pass-through gradient.
//
// Both give one CTA to one token row at a time (persistent over rows): the
// HBM traffic is one read of every input row and one write of every output
// row. The statistics are two-pass fp32 (mean first, then the mean of squared
// deviations), summed in a fixed order, so results are reproducible.
//
// Rows whose length is a multiple of 8 live in registers: each of THREADS
// threads holds C chunks of 8 elements, sized so that THREADS * C * 8 covers
// D. All loads of a row are issued before any of them is used, and the
// forward kernel issues the next row's loads before it reduces the current
// one, so each SM keeps 100+ KB of reads in flight (HBM needs about
// bandwidth x latency / SMs = 7 TB/s x 1.5 us / 152 = 70 KB). Other lengths
// use the shared-memory kernels (one row staged as fp32).
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

// Sum over a CTA of THREADS threads; every thread gets the result. `red`
// holds 32 floats.
template <int THREADS>
__device__ __forceinline__ float block_sum_t(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();  // the previous call's readers are done with `red`
  if (l == 0) red[w] = v;
  __syncthreads();
  return warp_sum(l < (THREADS >> 5) ? red[l] : 0.f);
}

// Two sums in one round of barriers; `red` holds 64 floats.
template <int THREADS>
__device__ __forceinline__ void block_sum2_t(float& a, float& b, float* red) {
  a = warp_sum(a);
  b = warp_sum(b);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) {
    red[w] = a;
    red[32 + w] = b;
  }
  __syncthreads();
  a = warp_sum(l < (THREADS >> 5) ? red[l] : 0.f);
  b = warp_sum(l < (THREADS >> 5) ? red[32 + l] : 0.f);
}

__device__ __forceinline__ float block_sum(float v, float* red) { return block_sum_t<kRowThreads>(v, red); }

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

// ------------------------------------------------------------ rows in registers

// 8 elements of E as loaded (16 bytes of bf16, 32 bytes of fp32).
template <typename E>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  uint4 w;
};
template <>
struct Raw8<float> {
  float4 a, b;
};

__device__ __forceinline__ void ld8(const __nv_bfloat16* p, Raw8<__nv_bfloat16>& r) {
  r.w = __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void ld8(const float* p, Raw8<float>& r) {
  r.a = __ldcs(reinterpret_cast<const float4*>(p));
  r.b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
}
__device__ __forceinline__ void zero8(Raw8<__nv_bfloat16>& r) { r.w = make_uint4(0, 0, 0, 0); }
__device__ __forceinline__ void zero8(Raw8<float>& r) { r.a = r.b = make_float4(0.f, 0.f, 0.f, 0.f); }
__device__ __forceinline__ void unpack8(const Raw8<__nv_bfloat16>& r, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r.w);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 t = __bfloat1622float2(h[j]);
    f[2 * j] = t.x;
    f[2 * j + 1] = t.y;
  }
}
__device__ __forceinline__ void unpack8(const Raw8<float>& r, float (&f)[8]) {
  f[0] = r.a.x, f[1] = r.a.y, f[2] = r.a.z, f[3] = r.a.w, f[4] = r.b.x, f[5] = r.b.y, f[6] = r.b.z, f[7] = r.b.w;
}

// Chunk k of this thread is chunk threadIdx.x + k * THREADS of the row;
// chunks past the row's nch load as zeros.
template <typename E, int THREADS, int C>
__device__ __forceinline__ void fetch_row(const E* __restrict__ row, int nch, Raw8<E> (&r)[C]) {
#pragma unroll
  for (int k = 0; k < C; ++k) {
    const int c = threadIdx.x + k * THREADS;
    if (c < nch)
      ld8(row + 8 * c, r[k]);
    else
      zero8(r[k]);
  }
}

// Layer norm of rows of D = 8 * nch elements held as C chunks per thread;
// the next row's loads are issued before the current row is reduced.
template <typename E, int THREADS, int C>
__global__ void __launch_bounds__(THREADS) layer_norm_reg_kernel(const E* __restrict__ x, int64_t T, int D, float eps,
                                                                 E* __restrict__ y) {
  __shared__ float red[32];
  pdl_wait();
  pdl_launch_dependents();
  const int nch = D >> 3;
  Raw8<E> nxt[C];
  int64_t t = blockIdx.x;
  if (t < T) fetch_row<E, THREADS, C>(x + t * D, nch, nxt);
  for (; t < T; t += gridDim.x) {
    float v[C][8];
#pragma unroll
    for (int k = 0; k < C; ++k) unpack8(nxt[k], v[k]);
    if (t + gridDim.x < T) fetch_row<E, THREADS, C>(x + (t + gridDim.x) * D, nch, nxt);
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < C; ++k)
#pragma unroll
      for (int j = 0; j < 8; ++j) s += v[k][j];  // zero-filled chunks add nothing
    const float mean = block_sum_t<THREADS>(s, red) / static_cast<float>(D);
    float q = 0.f;
#pragma unroll
    for (int k = 0; k < C; ++k) {
      if (static_cast<int>(threadIdx.x) + k * THREADS >= nch) continue;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float d = v[k][j] - mean;
        q += d * d;
      }
    }
    const float r = 1.0f / sqrtf(block_sum_t<THREADS>(q, red) / static_cast<float>(D) + eps);
    E* yr = y + t * D;
#pragma unroll
    for (int k = 0; k < C; ++k) {
      const int c = threadIdx.x + k * THREADS;
      if (c >= nch) continue;
      float f[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] = (v[k][j] - mean) * r;
      store8(yr + 8 * c, f);
    }
  }
}

// The backward tail with one chunk per thread (D = 8 * nch <= 8 * THREADS):
// x, dout and every partial of the thread's chunk are loaded before they are
// combined (partials two at a time, added in shard order).
template <typename E, int THREADS>
__global__ void __launch_bounds__(THREADS) layer_norm_bwd_reg_kernel(const float* __restrict__ G, int n,
                                                                     const E* __restrict__ x,
                                                                     const E* __restrict__ dout, int64_t T, int D,
                                                                     float eps, float* __restrict__ dx) {
  __shared__ float red[64];
  pdl_wait();
  pdl_launch_dependents();
  const int nch = D >> 3;
  const int c = threadIdx.x;
  const bool on = c < nch;
  const int64_t gstride = T * D;
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    const int64_t at = t * D + 8 * c;
    Raw8<E> xr, dr;
    float g[8], v[8];
    if (on) {
      ld8(x + at, xr);
      ld8(dout + at, dr);
      load8(G + at, g);
      for (int k = 1; k < n; k += 2) {
        float a[8], b[8];
        load8(G + k * gstride + at, a);
        if (k + 1 < n) load8(G + (k + 1) * gstride + at, b);
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] += a[j];
        if (k + 1 < n) {
#pragma unroll
          for (int j = 0; j < 8; ++j) g[j] += b[j];
        }
      }
      unpack8(xr, v);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) g[j] = v[j] = 0.f;
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += v[j];
    const float mean = block_sum_t<THREADS>(s, red) / static_cast<float>(D);
    float q = 0.f;
    if (on) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float d = v[j] - mean;
        q += d * d;
      }
    }
    const float r = 1.0f / sqrtf(block_sum_t<THREADS>(q, red) / static_cast<float>(D) + eps);
    float sg = 0.f, sgy = 0.f;
    if (on) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[j] = (v[j] - mean) * r;  // y
        sg += g[j];
        sgy += g[j] * v[j];
      }
    }
    block_sum2_t<THREADS>(sg, sgy, red);
    const float mg = sg / static_cast<float>(D), mgy = sgy / static_cast<float>(D);
    if (on) {
      float d[8], f[8];
      unpack8(dr, d);
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] = d[j] + r * (g[j] - mg - v[j] * mgy);
      store8(dx + at, f);
    }
  }
}

// out[j] += res[j] (fp32), for the fp32 path's fused sum.
__global__ void add_residual_f32_kernel(float* __restrict__ out, const float* __restrict__ res, int64_t count) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t j = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; j < count; j += stride) out[j] = out[j] + res[j];
}

template <typename K>
int row_grid(K kern, int threads, size_t smem, int64_t T) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int64_t cap = int64_t(num_sms()) * per_sm;
  return static_cast<int>(T < cap ? T : cap);
}

template <typename K>
cudaError_t set_smem(K kern, size_t smem) {
  if (smem <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
}

// Smallest power of two >= v, within [32, 1024].
int pow2_threads(int v) {
  int t = 32;
  while (t < v && t < 1024) t <<= 1;
  return t;
}

template <typename E, int THREADS, int C>
cudaError_t ln_reg(const E* x, int64_t T, int D, float eps, E* y, cudaStream_t s) {
  auto k = layer_norm_reg_kernel<E, THREADS, C>;
  return launch_pdl(k, dim3(row_grid(k, THREADS, 0, T)), dim3(THREADS), 0, s, x, T, D, eps, y);
}

// Forward: two chunks per thread where the row allows (so each thread has
// four 16-byte loads in flight with the next row's), else one.
template <typename E>
cudaError_t ln_dispatch(const E* x, int64_t T, int D, float eps, E* y, cudaStream_t s) {
  const int nch = D / 8;
  const int threads = pow2_threads((nch + 1) / 2);
  const int C = (nch + threads - 1) / threads;
  if (D % 8 == 0 && C <= 2) {
#define TPMLP_LN_CASE(TH)                                                        \
  case TH:                                                                       \
    return C == 1 ? ln_reg<E, TH, 1>(x, T, D, eps, y, s) : ln_reg<E, TH, 2>(x, T, D, eps, y, s);
    switch (threads) {
      TPMLP_LN_CASE(32)
      TPMLP_LN_CASE(64)
      TPMLP_LN_CASE(128)
      TPMLP_LN_CASE(256)
      TPMLP_LN_CASE(512)
      TPMLP_LN_CASE(1024)
      default:
        break;
    }
#undef TPMLP_LN_CASE
  }
  const size_t smem = (32 + size_t(D)) * sizeof(float);
  auto k = layer_norm_kernel<E>;
  cudaError_t e = set_smem(k, smem);
  if (e != cudaSuccess) return e;
  k<<<row_grid(k, kRowThreads, smem, T), kRowThreads, smem, s>>>(x, T, D, eps, y);
  return cudaGetLastError();
}

template <typename E, int THREADS>
cudaError_t lnb_reg(const float* G, int n, const E* x, const E* dout, int64_t T, int D, float eps, float* dx,
                    cudaStream_t s) {
  auto k = layer_norm_bwd_reg_kernel<E, THREADS>;
  return launch_pdl(k, dim3(row_grid(k, THREADS, 0, T)), dim3(THREADS), 0, s, G, n, x, dout, T, D, eps, dx);
}

// Backward tail: one chunk per thread up to D = 8192, else the shared-memory kernel.
template <typename E>
cudaError_t lnb_dispatch(const float* G, int n, const E* x, const E* dout, int64_t T, int D, float eps, float* dx,
                         cudaStream_t s) {
  const int nch = D / 8;
  if (D % 8 == 0 && nch <= 1024) {
    switch (pow2_threads(nch)) {
      case 32:
        return lnb_reg<E, 32>(G, n, x, dout, T, D, eps, dx, s);
      case 64:
        return lnb_reg<E, 64>(G, n, x, dout, T, D, eps, dx, s);
      case 128:
        return lnb_reg<E, 128>(G, n, x, dout, T, D, eps, dx, s);
      case 256:
        return lnb_reg<E, 256>(G, n, x, dout, T, D, eps, dx, s);
      case 512:
        return lnb_reg<E, 512>(G, n, x, dout, T, D, eps, dx, s);
      default:
        return lnb_reg<E, 1024>(G, n, x, dout, T, D, eps, dx, s);
    }
  }
  const size_t smem = (32 + 2 * size_t(D)) * sizeof(float);
  auto k = layer_norm_bwd_kernel<E>;
  cudaError_t e = set_smem(k, smem);
  if (e != cudaSuccess) return e;
  k<<<row_grid(k, kRowThreads, smem, T), kRowThreads, smem, s>>>(G, n, x, dout, T, D, eps, dx);
  return cudaGetLastError();
}

}  // namespace

size_t layer_norm_max_d() { return (200 * 1024) / 8 - 64; }

cudaError_t launch_layer_norm(const void* x, int64_t T, int D, float eps, int is_bf16, void* y, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (is_bf16)
    return ln_dispatch(static_cast<const __nv_bfloat16*>(x), T, D, eps, static_cast<__nv_bfloat16*>(y), s);
  return ln_dispatch(static_cast<const float*>(x), T, D, eps, static_cast<float*>(y), s);
}

cudaError_t launch_layer_norm_bwd(const float* G, int n, const void* x, const void* dout, int64_t T, int D, float eps,
                                  int is_bf16, float* dx, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (is_bf16)
    return lnb_dispatch(G, n, static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(dout), T, D,
                        eps, dx, s);
  return lnb_dispatch(G, n, static_cast<const float*>(x), static_cast<const float*>(dout), T, D, eps, dx, s);
}

cudaError_t launch_add_residual_f32(float* out, const float* res, int64_t count, cudaStream_t s) {
  if (count <= 0) return cudaSuccess;
  const int64_t want = (count + kRowThreads - 1) / kRowThreads;
  const int64_t cap = int64_t(num_sms()) * 8;
  add_residual_f32_kernel<<<static_cast<int>(want < cap ? want : cap), kRowThreads, 0, s>>>(out, res, count);
  return cudaGetLastError();
}

}  // namespace tpmlp
