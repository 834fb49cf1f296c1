// elementwise.cu — the memory-bound kernels of the path: standalone GeLU, the
// shard-ordered partial-sum reduction (the simulated all-reduce), the shard
// slicing copies, 2-byte transposes, the backward activation step, and the
// bounded-wait self test.
#include "device.cuh"
#include "internal.h"

namespace tpmlp {

namespace {

constexpr int kEwThreads = 256;

int ew_grid(int64_t work_items, int per_thread) {
  const int64_t want = (work_items + int64_t(kEwThreads) * per_thread - 1) / (int64_t(kEwThreads) * per_thread);
  const int64_t cap = int64_t(num_sms()) * 8;  // 8 resident blocks of 256 per SM
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

// ------------------------------------------------------------------ GeLU

__global__ void gelu_f32_kernel(const float* __restrict__ x, float* __restrict__ y, int64_t n) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t n4 = n / 4;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 v = reinterpret_cast<const float4*>(x)[i];
    v.x = gelu_fast(v.x);
    v.y = gelu_fast(v.y);
    v.z = gelu_fast(v.z);
    v.w = gelu_fast(v.w);
    reinterpret_cast<float4*>(y)[i] = v;
  }
  for (int64_t i = n4 * 4 + int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) y[i] = gelu_fast(x[i]);
}

__global__ void gelu_bf16_kernel(const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ y, int64_t n) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t n8 = n / 8;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    uint4 w = reinterpret_cast<const uint4*>(x)[i];
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 f = __bfloat1622float2(h[j]);
      h[j] = __floats2bfloat162_rn(gelu_fast(f.x), gelu_fast(f.y));
    }
    reinterpret_cast<uint4*>(y)[i] = w;
  }
  for (int64_t i = n8 * 8 + int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    y[i] = __float2bfloat16_rn(gelu_fast(__bfloat162float(x[i])));
}

// ------------------------------------------------------------------ all-reduce

// Y[j] = ((Yp[0][j] + Yp[1][j]) + Yp[2][j]) + ... in fp32, shard order fixed,
// and with a residual R (res_kind 1: fp32, 2: bf16) then Y[j] = R[j] + that
// sum. Each thread owns float4 columns of the [n][count] block; the n loads of
// one float4 are issued before the adds so n*16 bytes per thread are in
// flight. Partials are read once (streaming loads), Y is written once.
__device__ __forceinline__ float4 residual4(const void* res, int res_kind, int64_t i) {
  if (res_kind == 1) return __ldcs(reinterpret_cast<const float4*>(res) + i);
  const uint2 w = __ldcs(reinterpret_cast<const uint2*>(res) + i);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ float residual1(const void* res, int res_kind, int64_t j) {
  if (res_kind == 1) return static_cast<const float*>(res)[j];
  return __bfloat162float(static_cast<const __nv_bfloat16*>(res)[j]);
}

// The output is cut into gridDim.y equal row slices (the ranks of a
// reduce-scatter; one slice for the all-reduce): blocks with blockIdx.y = j
// handle the `slice` elements j*slice .. (j+1)*slice - 1 and write them to
// out.p[j].
template <int NMAX>
__global__ void __launch_bounds__(kEwThreads) allreduce_kernel(const float* __restrict__ Yp, int n, int64_t count,
                                                               const void* __restrict__ res, int res_kind,
                                                               OutSlices out, int* status) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t slice = count / gridDim.y;
  const int64_t base4 = int64_t(blockIdx.y) * (slice / 4);
  float* __restrict__ Y = out.p[blockIdx.y];
  const int64_t n4 = slice / 4;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const float4* P = reinterpret_cast<const float4*>(Yp) + base4;
  const int64_t shard_stride4 = count / 4;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    if (!TPMLP_DCHECK(base4 + i < count / 4 && Y != nullptr, status, kChkReduce)) break;
    float4 v[NMAX];
#pragma unroll
    for (int s = 0; s < NMAX; ++s)
      if (s < n) v[s] = __ldcs(P + s * shard_stride4 + i);
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
    if (res_kind) r = residual4(res, res_kind, base4 + i);
    float4 acc = v[0];
#pragma unroll
    for (int s = 1; s < NMAX; ++s) {
      if (s < n) {
        acc.x += v[s].x;
        acc.y += v[s].y;
        acc.z += v[s].z;
        acc.w += v[s].w;
      }
    }
    if (res_kind) {
      acc.x = r.x + acc.x;
      acc.y = r.y + acc.y;
      acc.z = r.z + acc.z;
      acc.w = r.w + acc.w;
    }
    __stcs(reinterpret_cast<float4*>(Y) + i, acc);
  }
}

// Any n and any slice length: the same order, shards taken from memory one by one.
__global__ void allreduce_any_kernel(const float* __restrict__ Yp, int n, int64_t count, const void* __restrict__ res,
                                     int res_kind, OutSlices out, int* status) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t slice = count / gridDim.y;
  const int64_t base = int64_t(blockIdx.y) * slice;
  float* __restrict__ Y = out.p[blockIdx.y];
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t j = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; j < slice; j += stride) {
    if (!TPMLP_DCHECK(base + j < count && Y != nullptr, status, kChkReduce)) break;
    float acc = Yp[base + j];
    for (int s = 1; s < n; ++s) acc += Yp[int64_t(s) * count + base + j];
    Y[j] = res_kind ? residual1(res, res_kind, base + j) + acc : acc;
  }
}

// ------------------------------------------------------------------ all-gather

// out = the n input slices back to back (slice_bytes each), blockIdx.y = slice.
// Each thread moves eight words per pass, all eight loads issued first; the
// output is written with the streaming (evict-first) hint like the reduce's.
template <typename W>
__global__ void gather_slices_kernel(InSlices in, int64_t words, W* __restrict__ out, int* status) {
  pdl_wait();
  pdl_launch_dependents();
  if (!TPMLP_DCHECK(blockIdx.y < kMaxGroups && in.p[blockIdx.y] != nullptr, status, kChkReduce)) return;
  const W* __restrict__ src = static_cast<const W*>(in.p[blockIdx.y]);
  W* __restrict__ dst = out + int64_t(blockIdx.y) * words;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 7 * stride < words; i += 8 * stride) {
    W w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = __ldcs(src + i + k * stride);
#pragma unroll
    for (int k = 0; k < 8; ++k) __stcs(dst + i + k * stride, w[k]);
  }
  for (; i < words; i += stride) __stcs(dst + i, __ldcs(src + i));
}

// ------------------------------------------------------------------ shard copies

// A_i[r, c] = A[r, f0 + c] and B_i[r, c] = B[f0 + r, c]; one element per thread
// step, grid-stride over the D*F elements of A and of B. Every shard reads its
// destinations from the device descriptor table.
template <typename E>
__global__ void shard_copy_kernel(const E* __restrict__ A, const E* __restrict__ B, const ShardDesc* __restrict__ tab,
                                  int64_t D, int64_t F, int64_t Fs) {
  const int64_t total = D * F;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total; e += stride) {
    {  // A: element (r, f) of [D, F]
      const int64_t r = e / F, f = e % F;
      const int64_t i = f / Fs, c = f % Fs;
      static_cast<E*>(tab[i].A)[r * Fs + c] = A[e];
    }
    {  // B: element (f, c) of [F, D]
      const int64_t f = e / D, c = e % D;
      const int64_t i = f / Fs, r = f % Fs;
      static_cast<E*>(tab[i].B)[r * D + c] = B[e];
    }
  }
}

// ------------------------------------------------------------------ transpose

// out[c, r] = in[r, c] for 2-byte elements, 64 x 64 tiles through shared memory.
__global__ void __launch_bounds__(256) transpose_u16_kernel(const uint16_t* __restrict__ in, int64_t rows,
                                                            int64_t cols, int64_t ldi, uint16_t* __restrict__ out,
                                                            int64_t ldo) {
  __shared__ uint16_t tile[64][66];
  const int64_t r0 = int64_t(blockIdx.y) * 64, c0 = int64_t(blockIdx.x) * 64;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  // Read 64 rows x 64 columns: each thread moves 2 adjacent columns per row.
  for (int rr = ty; rr < 64; rr += 8) {
    const int64_t r = r0 + rr, c = c0 + 2 * tx;
    uint16_t a = 0, b = 0;
    if (r < rows) {
      if (c < cols) a = in[r * ldi + c];
      if (c + 1 < cols) b = in[r * ldi + c + 1];
    }
    tile[rr][2 * tx] = a;
    tile[rr][2 * tx + 1] = b;
  }
  __syncthreads();
  for (int cc = ty; cc < 64; cc += 8) {
    const int64_t c = c0 + cc, r = r0 + 2 * tx;
    if (c < cols) {
      if (r < rows) out[c * ldo + r] = tile[2 * tx][cc];
      if (r + 1 < rows) out[c * ldo + r + 1] = tile[2 * tx + 1][cc];
    }
  }
}

// ------------------------------------------------------------------ backward activation (fp32 path)

// H <- GeLU(P) and, in place, dH <- dH * GeLU'(P); P is only read. (The bf16
// path applies this step in the epilogue of its dH product instead.)
__global__ void bwd_act_f32_kernel(const float* __restrict__ P, float* __restrict__ H, float* __restrict__ dH,
                                   int64_t count) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t j = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; j < count; j += stride) {
    float g, dg;
    gelu_and_grad_fast(P[j], g, dg);
    H[j] = g;
    dH[j] = dH[j] * dg;
  }
}

}  // namespace

cudaError_t launch_gelu(const void* x, void* y, int64_t n, int is_bf16, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (is_bf16) {
    gelu_bf16_kernel<<<ew_grid(n, 8), kEwThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(x),
                                                         static_cast<__nv_bfloat16*>(y), n);
  } else {
    gelu_f32_kernel<<<ew_grid(n, 4), kEwThreads, 0, s>>>(static_cast<const float*>(x), static_cast<float*>(y), n);
  }
  return cudaGetLastError();
}

cudaError_t launch_reduce_scatter(const float* Yp, int n, int64_t count, const OutSlices& out, int nslices,
                                  cudaStream_t s, const void* res, int res_kind) {
  if (count <= 0) return cudaSuccess;
  if (nslices < 1 || nslices > kMaxGroups || count % nslices != 0) return cudaErrorInvalidValue;
  if (!res) res_kind = 0;
  const int64_t slice = count / nslices;
  const unsigned gy = static_cast<unsigned>(nslices);
  if (slice % 4 != 0) {  // slices would not be 16-byte aligned
    dim3 g(static_cast<unsigned>((ew_grid(count, 1) + nslices - 1) / nslices), gy);
    return launch_pdl(allreduce_any_kernel, g, dim3(kEwThreads), 0, s, Yp, n, count, res, res_kind, out,
                      device_status_word());
  }
  dim3 g(static_cast<unsigned>((ew_grid(count, 4) + nslices - 1) / nslices), gy);
  const dim3 b(kEwThreads);
  int* st = device_status_word();
  if (n <= 4) return launch_pdl(allreduce_kernel<4>, g, b, 0, s, Yp, n, count, res, res_kind, out, st);
  if (n <= 8) return launch_pdl(allreduce_kernel<8>, g, b, 0, s, Yp, n, count, res, res_kind, out, st);
  if (n <= 16) return launch_pdl(allreduce_kernel<16>, g, b, 0, s, Yp, n, count, res, res_kind, out, st);
  return launch_pdl(allreduce_any_kernel, g, b, 0, s, Yp, n, count, res, res_kind, out, st);
}

cudaError_t launch_allreduce(const float* Yp, int n, int64_t count, float* Y, cudaStream_t s, const void* res,
                             int res_kind) {
  OutSlices out{};
  out.p[0] = Y;
  return launch_reduce_scatter(Yp, n, count, out, 1, s, res, res_kind);
}

cudaError_t launch_all_gather(const InSlices& in, int nslices, int64_t slice_bytes, void* out, cudaStream_t s) {
  if (slice_bytes <= 0) return cudaSuccess;
  if (nslices < 1 || nslices > kMaxGroups) return cudaErrorInvalidValue;
  const unsigned gy = static_cast<unsigned>(nslices);
  auto gx = [&](int64_t words) {
    return static_cast<unsigned>((ew_grid(words * nslices, 4) + nslices - 1) / nslices);
  };
  const dim3 b(kEwThreads);
  if (slice_bytes % 16 == 0) {
    const int64_t w = slice_bytes / 16;
    return launch_pdl(gather_slices_kernel<uint4>, dim3(gx(w), gy), b, 0, s, in, w, static_cast<uint4*>(out),
                      device_status_word());
  }
  if (slice_bytes % 4 == 0) {
    const int64_t w = slice_bytes / 4;
    return launch_pdl(gather_slices_kernel<uint32_t>, dim3(gx(w), gy), b, 0, s, in, w, static_cast<uint32_t*>(out),
                      device_status_word());
  }
  const int64_t w = slice_bytes / 2;
  return launch_pdl(gather_slices_kernel<uint16_t>, dim3(gx(w), gy), b, 0, s, in, w, static_cast<uint16_t*>(out),
                      device_status_word());
}

cudaError_t launch_shard_copy(const void* A, const void* B, const ShardDesc* d_table, int64_t D, int64_t F,
                              int64_t Fs, int elem_bytes, cudaStream_t s) {
  const int g = ew_grid(D * F, 1);
  if (elem_bytes == 2)
    shard_copy_kernel<uint16_t><<<g, kEwThreads, 0, s>>>(static_cast<const uint16_t*>(A),
                                                          static_cast<const uint16_t*>(B), d_table, D, F, Fs);
  else
    shard_copy_kernel<uint32_t><<<g, kEwThreads, 0, s>>>(static_cast<const uint32_t*>(A),
                                                          static_cast<const uint32_t*>(B), d_table, D, F, Fs);
  return cudaGetLastError();
}

cudaError_t launch_transpose_u16(const void* in, int64_t rows, int64_t cols, int64_t ldi, void* out, int64_t ldo,
                                 cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>((cols + 63) / 64), static_cast<unsigned>((rows + 63) / 64));
  transpose_u16_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(in), rows, cols, ldi,
                                            static_cast<uint16_t*>(out), ldo);
  return cudaGetLastError();
}

cudaError_t launch_bwd_act_f32(const float* P, float* H, float* dH, int64_t count, cudaStream_t s) {
  if (count <= 0) return cudaSuccess;
  bwd_act_f32_kernel<<<ew_grid(count, 1), kEwThreads, 0, s>>>(P, H, dH, count);
  return cudaGetLastError();
}

}  // namespace tpmlp
