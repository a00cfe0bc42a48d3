// Portable SIMT projection kernel (fp32 FMA).  Serves the fp32 workloads and
// is the row-invariant reference schedule: every output accumulates its K
// products one at a time in increasing k, whatever M is and whichever tile
// the row falls in, so a row's result never depends on the batch around it.
#include "common.cuh"

namespace dflash {

template <typename T>
struct ASrcT {
  const T* p[DFLASH_MAX_PICK];
  int seg;
  int64_t ld;
  __device__ __forceinline__ float at(int64_t m, int k) const {
    const int s = k / seg;
    return to_f(p[s][m * ld + (k - s * seg)]);
  }
};

constexpr int SB_M = 64, SB_N = 64, SB_K = 16;

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(ASrcT<T> A, const T* __restrict__ W,
                                                        int64_t ldw, float* __restrict__ C,
                                                        int64_t ldc, int64_t M, int N, int K,
                                                        int accumulate) {
  __shared__ float As[SB_K][SB_M + 4];
  __shared__ float Ws[SB_K][SB_N + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t m0 = (int64_t)blockIdx.y * SB_M;
  const int n0 = blockIdx.x * SB_N;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += SB_K) {
    for (int e = threadIdx.x; e < SB_M * SB_K; e += 256) {
      const int mm = e / SB_K, kk = e - mm * SB_K;
      const int64_t m = m0 + mm;
      const int k = k0 + kk;
      As[kk][mm] = (m < M && k < K) ? A.at(m, k) : 0.f;
    }
    for (int e = threadIdx.x; e < SB_N * SB_K; e += 256) {
      const int nn = e / SB_K, kk = e - nn * SB_K;
      const int n = n0 + nn;
      const int k = k0 + kk;
      Ws[kk][nn] = (n < N && k < K) ? to_f(W[(int64_t)n * ldw + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SB_K; ++kk) {
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = Ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      float* c = C + m * ldc + n;
      *c = accumulate ? (*c + acc[i][j]) : acc[i][j];
    }
  }
}

// The same product for at most 16 rows (decode, verify, draft blocks): one
// output per thread, a CTA covering 16 rows x 16 columns, so N / 16 CTAs
// share the work instead of N / 64; K advances 64 at a time through shared
// memory, with the next K slice loaded into registers while the current one
// is used.  Each output is the same fmaf chain in increasing k as above, so
// the two kernels give identical bits for a row.
constexpr int SR_K = 64;

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_rows_kernel(ASrcT<T> A, const T* __restrict__ W,
                                                             int64_t ldw, float* __restrict__ C,
                                                             int64_t ldc, int M, int N, int K,
                                                             int accumulate) {
  __shared__ float As[16][SR_K + 1];
  __shared__ float Ws[16][SR_K + 1];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int n0 = blockIdx.x * 16;
  float ra[4], rw[4];
  auto load = [&](int k0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e = tid + q * 256, r = e / SR_K, k = k0 + (e - r * SR_K);
      ra[q] = (r < M && k < K) ? A.at(r, k) : 0.f;
      rw[q] = (n0 + r < N && k < K) ? to_f(W[(int64_t)(n0 + r) * ldw + k]) : 0.f;
    }
  };
  float acc = 0.f;
  load(0);
  for (int k0 = 0; k0 < K; k0 += SR_K) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e = tid + q * 256, r = e / SR_K, kk = e - r * SR_K;
      As[r][kk] = ra[q];
      Ws[r][kk] = rw[q];
    }
    __syncthreads();
    if (k0 + SR_K < K) load(k0 + SR_K);
    const int kn = min(SR_K, K - k0);
    for (int kk = 0; kk < kn; ++kk) acc = fmaf(As[ty][kk], Ws[tx][kk], acc);
    __syncthreads();
  }
  const int n = n0 + tx;
  if (ty < M && n < N) {
    float* c = C + (int64_t)ty * ldc + n;
    *c = accumulate ? (*c + acc) : acc;
  }
}

int gemm(dflash_handle* h, cudaStream_t s, int kclass, int dtype, const ASrc& A, const void* W,
         int64_t ldw, float* C, int64_t ldc, int64_t M, int N, int K, bool accumulate) {
  if (M <= 0 || N <= 0) return DFLASH_OK;
  const dim3 grid((N + SB_N - 1) / SB_N, (unsigned)((M + SB_M - 1) / SB_M));
  Timer t;
  launch_begin(h, kclass, s, &t);
  if (M <= 16) {
    const dim3 g2((N + 15) / 16);
    if (dtype == DFLASH_BF16) {
      ASrcT<bf16> a;
      for (int i = 0; i < DFLASH_MAX_PICK; ++i) a.p[i] = (const bf16*)A.p[i];
      a.seg = A.seg;
      a.ld = A.ld;
      gemm_simt_rows_kernel<bf16><<<g2, 256, 0, s>>>(a, (const bf16*)W, ldw, C, ldc, (int)M, N, K,
                                                     accumulate ? 1 : 0);
    } else {
      ASrcT<float> a;
      for (int i = 0; i < DFLASH_MAX_PICK; ++i) a.p[i] = (const float*)A.p[i];
      a.seg = A.seg;
      a.ld = A.ld;
      gemm_simt_rows_kernel<float><<<g2, 256, 0, s>>>(a, (const float*)W, ldw, C, ldc, (int)M, N,
                                                      K, accumulate ? 1 : 0);
    }
    return launch_end(h, s, &t);
  }
  if (dtype == DFLASH_BF16) {
    ASrcT<bf16> a;
    for (int i = 0; i < DFLASH_MAX_PICK; ++i) a.p[i] = (const bf16*)A.p[i];
    a.seg = A.seg;
    a.ld = A.ld;
    gemm_simt_kernel<bf16><<<grid, 256, 0, s>>>(a, (const bf16*)W, ldw, C, ldc, M, N, K,
                                                accumulate ? 1 : 0);
  } else {
    ASrcT<float> a;
    for (int i = 0; i < DFLASH_MAX_PICK; ++i) a.p[i] = (const float*)A.p[i];
    a.seg = A.seg;
    a.ld = A.ld;
    gemm_simt_kernel<float><<<grid, 256, 0, s>>>(a, (const float*)W, ldw, C, ldc, M, N, K,
                                                 accumulate ? 1 : 0);
  }
  return launch_end(h, s, &t);
}

}  // namespace dflash
