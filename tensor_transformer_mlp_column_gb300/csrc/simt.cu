// simt.cu — fp32 CUDA-core GEMM for the fp32 path (TPMLP_F32).
//
// The tensor cores' reduced-precision kinds cannot meet the fp32 accuracy the
// fp32 path promises, so fp32 products run as FFMA on the CUDA cores. Operands
// take arbitrary element strides, which covers every transpose the forward and
// backward passes need without copies. Tiles of 64 x 64 outputs, 256 threads,
// 4 x 4 outputs per thread, K staged through shared memory 16 at a time.
#include "device.cuh"
#include "internal.h"

namespace tpmlp {

namespace {

constexpr int TM = 64, TN = 64, TK = 16;

__global__ void __launch_bounds__(256) simt_gemm_kernel(const SimtGemm g) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int tid = threadIdx.x;
  const int tr = tid / 16, tc = tid % 16;  // 16 x 16 threads, 4 x 4 outputs each
  const int64_t m0 = int64_t(blockIdx.y) * TM, n0 = int64_t(blockIdx.x) * TN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < g.K; k0 += TK) {
    // 64 x 16 of A and 16 x 64 of B: 1024 elements each, 4 per thread.
    for (int e = tid; e < TM * TK; e += 256) {
      const int mm = e / TK, kk = e % TK;
      const int64_t m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < g.M && k < g.K) ? g.A[m * g.sam + k * g.sak] : 0.f;
    }
    for (int e = tid; e < TK * TN; e += 256) {
      const int kk = e / TN, nn = e % TN;
      const int64_t k = k0 + kk, n = n0 + nn;
      Bs[kk][nn] = (k < g.K && n < g.N) ? g.B[k * g.sbk + n * g.sbn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][tr * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tc * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + tr * 4 + i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tc * 4 + j;
      if (n >= g.N) continue;
      float* c = g.C + m * g.ldc + n;
      if (g.epi == kSimtGelu)
        *c = gelu_fast(acc[i][j]);
      else if (g.epi == kSimtAccumulate)
        *c += acc[i][j];
      else
        *c = acc[i][j];
    }
  }
}

}  // namespace

cudaError_t launch_simt_gemm(const SimtGemm& g, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>((g.N + TN - 1) / TN), static_cast<unsigned>((g.M + TM - 1) / TM));
  simt_gemm_kernel<<<grid, 256, 0, s>>>(g);
  return cudaGetLastError();
}

}  // namespace tpmlp
