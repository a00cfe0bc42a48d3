// DFlash 2's grouped dynamic causal conv (txtmix source reading §13-§14):
// two taps, depthwise, over the rows of each block; every coefficient is a
// learned base kernel plus a correction projected from the row, one per
// group of channels.  conv_corr computes the corrections, conv_apply one
// call of the conv (prepare: into a separate buffer; finish: added into
// the residual).
#include "common.cuh"

namespace dflash {

// corr[r][j] = sum_d x[r][d] kp[j][d] (fp32 accumulation): one warp per
// (row, j), lanes over d.
template <typename T>
__global__ void __launch_bounds__(256) conv_corr_kernel(const float* __restrict__ x,
                                                        const T* __restrict__ kp, int D, int J,
                                                        float* __restrict__ corr) {
  const int lane = threadIdx.x & 31, j = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t r = blockIdx.y;
  if (j >= J) return;
  const float* xr = x + r * D;
  const T* w = kp + (int64_t)j * D;
  float acc = 0.f;
  for (int d = lane; d < D; d += 32) acc = fmaf(xr[d], to_f(w[d]), acc);
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) corr[r * J + j] = acc;
}

// out[r][c] (= or +=) k0 y[r][c] + k1 y[r-1][c], with k_tap = base[call][tap][c]
// + corr[r][call][tap][c / group] and no predecessor for a block's first row
// (r % B == 0).  y and out do not overlap.
__global__ void __launch_bounds__(256) conv_apply_kernel(const float* __restrict__ y,
                                                         const float* __restrict__ corr,
                                                         const float* __restrict__ base, int call,
                                                         int group, int D, int B, int64_t total,
                                                         float* __restrict__ out, int accumulate) {
  const int ng = D / group;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / D;
    const int c = (int)(e - r * D);
    const float* cr = corr + r * 4 * ng + call * 2 * ng + c / group;
    const float k0 = base[(call * 2) * D + c] + cr[0];
    const float k1 = base[(call * 2 + 1) * D + c] + cr[ng];
    float v = k0 * y[e];
    if (r % B != 0) v = fmaf(k1, y[e - D], v);
    out[e] = accumulate ? out[e] + v : v;
  }
}

int conv_corr(dflash_handle* h, cudaStream_t s, const float* x, const void* kp, int64_t R,
              float* corr) {
  const dflash_config& c = h->cfg;
  const int D = c.hidden, J = 4 * D / c.conv_group;
  const dim3 grid((J + 7) / 8, (unsigned)R);
  Timer t;
  launch_begin(h, DFLASH_K_ELEMENTWISE, s, &t);
  if (c.dtype == DFLASH_BF16)
    conv_corr_kernel<bf16><<<grid, 256, 0, s>>>(x, (const bf16*)kp, D, J, corr);
  else
    conv_corr_kernel<float><<<grid, 256, 0, s>>>(x, (const float*)kp, D, J, corr);
  return launch_end(h, s, &t);
}

int conv_apply(dflash_handle* h, cudaStream_t s, const float* y, const float* corr,
               const float* base, int call, int64_t R, int B, float* out, bool accumulate) {
  const dflash_config& c = h->cfg;
  const int64_t total = R * c.hidden;
  const int blocks = (int)std::min<int64_t>((total + 255) / 256, 4 * 152 * 8);
  Timer t;
  launch_begin(h, DFLASH_K_ELEMENTWISE, s, &t);
  conv_apply_kernel<<<blocks, 256, 0, s>>>(y, corr, base, call, c.conv_group, c.hidden, B, total,
                                          out, accumulate ? 1 : 0);
  return launch_end(h, s, &t);
}

}  // namespace dflash
