// hgemm_generic.cu — C = A·B for operands that TMA cannot describe (a base
// pointer not 16-byte aligned, or K or N not a multiple of 8, so that a row
// pitch is not a multiple of 16 bytes).
//
// Same arithmetic contract as the tensor-core path: FP16 inputs, FP32
// accumulation ("GPU架构与CUDA", 混合精度核函数), one round-to-nearest-even to
// FP16. Edge handling follows "GPU架构与CUDA", 共享内存与分块: tiles are staged
// in shared memory with out-of-range elements replaced by zero, and only
// in-range outputs are stored. Each FP16 product is exact in FP32, so every
// step here is an FP32 add of an exact product.
//
// Layout of the work: a 64×64 output tile per 256-thread block, K staged 32
// at a time; each thread owns a 4×4 patch of the tile.
#include <cuda_fp16.h>

#include "internal.h"

namespace hg {
namespace {

constexpr int GT_M = 64, GT_N = 64, GT_K = 32;

__global__ void __launch_bounds__(256)
    hgemm_generic_kernel(const uint16_t* __restrict__ A, const uint16_t* __restrict__ B,
                         uint16_t* __restrict__ C, int64_t M, int64_t N, int64_t K,
                         int64_t tiles_n) {
  // sA[k][i] and sB[k][j]: K-major staging, padded against bank conflicts
  __shared__ float sA[GT_K][GT_M + 4];
  __shared__ float sB[GT_K][GT_N + 4];
  const int64_t m0 = static_cast<int64_t>(blockIdx.x / tiles_n) * GT_M;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x % tiles_n) * GT_N;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int64_t k0 = 0; k0 < K; k0 += GT_K) {
    for (int e = threadIdx.x; e < GT_M * GT_K; e += 256) {
      const int r = e / GT_K, kk = e % GT_K;
      const int64_t gi = m0 + r, gk = k0 + kk;
      sA[kk][r] = (gi < M && gk < K) ? __half2float(__ushort_as_half(A[gi * K + gk])) : 0.f;
      const int64_t gj = n0 + r;
      sB[kk][r] = (gj < N && gk < K) ? __half2float(__ushort_as_half(B[gj * K + gk])) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < GT_K; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        a[u] = sA[kk][ty * 4 + u];
        b[u] = sB[kk][tx * 4 + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = __fmaf_rn(a[u], b[v], acc[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int64_t gi = m0 + ty * 4 + u;
    if (gi >= M) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int64_t gj = n0 + tx * 4 + v;
      if (gj < N) C[gi * N + gj] = __half_as_ushort(__float2half_rn(acc[u][v]));
    }
  }
}

}  // namespace

cudaError_t launch_generic(const PlainArgs& args, int /*num_sms*/, cudaStream_t stream) {
  const int64_t tiles_n = (args.N + GT_N - 1) / GT_N;
  const int64_t tiles = tiles_n * ((args.M + GT_M - 1) / GT_M);
  if (tiles > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  hgemm_generic_kernel<<<static_cast<unsigned>(tiles), 256, 0, stream>>>(
      args.A, args.B, args.C, args.M, args.N, args.K, tiles_n);
  return cudaGetLastError();
}

}  // namespace hg
