// Row-wise kernels of the draft path: block embedding, RMSNorm, per-head
// q/k norm + RoPE (+ store into a dense buffer or a K/V cache), SwiGLU, and
// cache-length bookkeeping.
#include "common.cuh"
#include "ptx.cuh"

namespace dflash {

// Block input rows [anchor, mask x (B-1)] through the shared embedding, times
// input_embedding_scale, into the fp32 residual stream (txtmix §6, §9).  All
// of a thread's loads are issued before the stores.
template <typename T>
__global__ void __launch_bounds__(256) embed_block_kernel(const T* __restrict__ E,
                                                          const int32_t* __restrict__ anchor,
                                                          int mask_id, int B, int V, int D,
                                                          float scale, float* __restrict__ x,
                                                          int* status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int r = blockIdx.x;
  const int b = r / B, i = r - b * B;
  const int id = (i == 0) ? anchor[b] : mask_id;
  float* dst = x + (int64_t)r * D;
  if (id < 0 || id >= V) {
    if (threadIdx.x == 0) atomicOr(status, ST_BOUNDS);
    for (int k = threadIdx.x; k < D; k += blockDim.x) dst[k] = 0.f;
    return;
  }
  const T* src = E + (int64_t)id * D;
  constexpr int C = 32;
  float v[C];
#pragma unroll
  for (int q = 0; q < C; ++q) {
    const int k = threadIdx.x + q * blockDim.x;
    v[q] = k < D ? to_f(src[k]) : 0.f;
  }
#pragma unroll
  for (int q = 0; q < C; ++q) {
    const int k = threadIdx.x + q * blockDim.x;
    if (k < D) dst[k] = v[q] * scale;
  }
  for (int k = threadIdx.x + C * blockDim.x; k < D; k += blockDim.x) dst[k] = to_f(src[k]) * scale;
}

template <typename T>
__global__ void embed_tokens_kernel(const T* __restrict__ E, const int32_t* __restrict__ tok, int V,
                                    int D, float scale, float* __restrict__ x, int* status) {
  const int r = blockIdx.x;
  const int id = tok[r];
  float* dst = x + (int64_t)r * D;
  if (id < 0 || id >= V) {
    if (threadIdx.x == 0) atomicOr(status, ST_BOUNDS);
    for (int k = threadIdx.x; k < D; k += blockDim.x) dst[k] = 0.f;
    return;
  }
  const T* src = E + (int64_t)id * D;
  for (int k = threadIdx.x; k < D; k += blockDim.x) dst[k] = to_f(src[k]) * scale;
}

// out[r] = in[r'] / sqrt(mean(in[r']^2) + eps) * g, fp32 arithmetic.
// skip_first_of > 1 maps output row r to input row r' that skips the first
// row of every group of skip_first_of rows (the anchor rows of a block).
// Each thread first loads all of its elements (up to RN_CACHE) into registers
// so the loads are in flight together, then reduces, then writes.
constexpr int RN_CACHE = 32;
template <typename TI, typename TO>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const TI* __restrict__ in, int64_t ld_in,
                                                      TO* __restrict__ out, int64_t ld_out,
                                                      const float* __restrict__ g, int D, float eps,
                                                      int skip_first_of) {
  __shared__ float red[33];
  // launched as a programmatic dependent: it may be resident while the kernel
  // before it finishes, and reads its input only after that kernel is done
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t r = blockIdx.x;
  int64_t ri = r;
  if (skip_first_of > 1) {
    const int64_t per = skip_first_of - 1;
    ri = (r / per) * skip_first_of + (r % per) + 1;
  }
  const TI* src = in + ri * ld_in;
  float v[RN_CACHE];
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < RN_CACHE; ++q) {
    const int k = threadIdx.x + q * blockDim.x;
    v[q] = (k < D) ? to_f(src[k]) : 0.f;
  }
#pragma unroll
  for (int q = 0; q < RN_CACHE; ++q) ss += v[q] * v[q];
  for (int k = threadIdx.x + RN_CACHE * blockDim.x; k < D; k += blockDim.x) {
    const float x = to_f(src[k]);
    ss += x * x;
  }
  ss = block_sum(ss, red);
  const float rinv = 1.0f / sqrtf(ss / (float)D + eps);
  TO* dst = out + r * ld_out;
#pragma unroll
  for (int q = 0; q < RN_CACHE; ++q) {
    const int k = threadIdx.x + q * blockDim.x;
    if (k < D) dst[k] = from_f<TO>(v[q] * rinv * g[k]);
  }
  for (int k = threadIdx.x + RN_CACHE * blockDim.x; k < D; k += blockDim.x)
    dst[k] = from_f<TO>(to_f(src[k]) * rinv * g[k]);
}

// One warp per (row, head): optional per-head RMSNorm, optional RoPE with
// rotate-half pairs (j, j + d/2), then store (dense or cache at len[b] + i).
template <typename T>
__global__ void head_norm_rope_kernel(const float* __restrict__ in, int64_t rows, int heads, int d,
                                      const float* __restrict__ gain, int use_rope, RowMap rm,
                                      const int32_t* __restrict__ len,
                                      const float2* __restrict__ rope_tab, int max_pos, float eps,
                                      T* dense, T* cache, int cap, int cache_batch, int* status) {
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= rows * heads) return;
  const int64_t r = warp / heads;
  const int hd = (int)(warp - r * heads);
  int b, i;
  if (!rm.map((int)r, b, i)) return;
  const int pos = len[b] + i;
  const float* src = in + r * (int64_t)(heads * d) + (int64_t)hd * d;
  const int half = d >> 1;
  const int P = half >> 5;           // pairs per lane: 1 (d = 64) or 2 (d = 128)
  float x1[2], x2[2];
  float ss = 0.f;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    if (p < P) {
      const int j = lane + 32 * p;
      x1[p] = src[j];
      x2[p] = src[j + half];
      ss += x1[p] * x1[p] + x2[p] * x2[p];
    }
  }
  if (gain != nullptr) {
    ss = warp_sum(ss);
    const float rinv = 1.0f / sqrtf(ss / (float)d + eps);
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      if (p < P) {
        const int j = lane + 32 * p;
        x1[p] = x1[p] * rinv * gain[j];
        x2[p] = x2[p] * rinv * gain[j + half];
      }
    }
  }
  if (use_rope) {
    if (pos < 0 || pos >= max_pos) {
      if (lane == 0) atomicOr(status, ST_BOUNDS);
      return;
    }
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      if (p < P) {
        const int j = lane + 32 * p;
        const float2 cs = rope_tab[(int64_t)pos * half + j];
        const float y1 = x1[p] * cs.x - x2[p] * cs.y;
        const float y2 = x2[p] * cs.x + x1[p] * cs.y;
        x1[p] = y1;
        x2[p] = y2;
      }
    }
  }
  T* dst;
  if (cache != nullptr) {
    if (b >= cache_batch || pos < 0 || pos >= cap) {
      if (lane == 0) atomicOr(status, ST_CAPACITY);
      return;
    }
    dst = cache + (((int64_t)b * heads + hd) * cap + pos) * d;
  } else {
    dst = dense + r * (int64_t)(heads * d) + (int64_t)hd * d;
  }
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    if (p < P) {
      const int j = lane + 32 * p;
      dst[j] = from_f<T>(x1[p]);
      dst[j + half] = from_f<T>(x2[p]);
    }
  }
}

// a = SiLU(g) * u, SiLU(x) = x / (1 + e^-x).
template <typename T>
__global__ void swiglu_kernel(const float* __restrict__ g, const float* __restrict__ u,
                              T* __restrict__ a, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float x = g[i];
    a[i] = from_f<T>(x / (1.0f + expf(-x)) * u[i]);
  }
}

template <typename T>
__global__ void cast_kernel(const float* __restrict__ in, T* __restrict__ out, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = from_f<T>(in[i]);
}

__global__ void advance_len_kernel(int32_t* len, const int32_t* nrows, int uniform, int batch,
                                   int cap, int* status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int n = nrows ? nrows[b] : uniform;
  if (n < 0 || len[b] + n > cap) {
    atomicOr(status, ST_CAPACITY);
    return;
  }
  len[b] += n;
}

// ---------------------------------------------------------------------------
int embed_block(dflash_handle* h, cudaStream_t s, int dtype, const void* E, const int32_t* anchor,
                int mask_id, int batch, int B, int V, int D, float scale, float* x) {
  Timer t;
  launch_begin(h, DFLASH_K_ELEMENTWISE, s, &t);
  if (dtype == DFLASH_BF16)
    embed_block_kernel<bf16><<<batch * B, 256, 0, s>>>((const bf16*)E, anchor, mask_id, B, V, D,
                                                       scale, x, h->d_status);
  else
    embed_block_kernel<float><<<batch * B, 256, 0, s>>>((const float*)E, anchor, mask_id, B, V, D,
                                                        scale, x, h->d_status);
  return launch_end(h, s, &t);
}

int embed_tokens(dflash_handle* h, cudaStream_t s, int dtype, const void* E, const int32_t* tok,
                 int rows, int V, int D, float scale, float* x) {
  Timer t;
  launch_begin(h, DFLASH_K_ELEMENTWISE, s, &t);
  if (dtype == DFLASH_BF16)
    embed_tokens_kernel<bf16><<<rows, 256, 0, s>>>((const bf16*)E, tok, V, D, scale, x, h->d_status);
  else
    embed_tokens_kernel<float><<<rows, 256, 0, s>>>((const float*)E, tok, V, D, scale, x,
                                                    h->d_status);
  return launch_end(h, s, &t);
}

int rmsnorm_rows(dflash_handle* h, cudaStream_t s, int in_dtype, int out_dtype, const void* in,
                 int64_t ld_in, void* out, int64_t ld_out, const float* g, int64_t rows, int D,
                 float eps, int skip_first_of) {
  if (rows <= 0) return DFLASH_OK;
  Timer t;
  launch_begin(h, DFLASH_K_ELEMENTWISE, s, &t);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)rows);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (in_dtype == DFLASH_F32 && out_dtype == DFLASH_F32)
    cudaLaunchKernelEx(&cfg, rmsnorm_kernel<float, float>, (const float*)in, ld_in, (float*)out,
                       ld_out, g, D, eps, skip_first_of);
  else if (in_dtype == DFLASH_F32 && out_dtype == DFLASH_BF16)
    cudaLaunchKernelEx(&cfg, rmsnorm_kernel<float, bf16>, (const float*)in, ld_in, (bf16*)out,
                       ld_out, g, D, eps, skip_first_of);
  else if (in_dtype == DFLASH_BF16 && out_dtype == DFLASH_BF16)
    cudaLaunchKernelEx(&cfg, rmsnorm_kernel<bf16, bf16>, (const bf16*)in, ld_in, (bf16*)out,
                       ld_out, g, D, eps, skip_first_of);
  else
    cudaLaunchKernelEx(&cfg, rmsnorm_kernel<bf16, float>, (const bf16*)in, ld_in, (float*)out,
                       ld_out, g, D, eps, skip_first_of);
  return launch_end(h, s, &t);
}

int head_norm_rope(dflash_handle* h, cudaStream_t s, int dtype, const float* in, int64_t rows,
                   int heads, int d, const float* gain, bool rope, const RowMap& rm,
                   const int32_t* len, void* dense, void* cache, int cap, int cache_batch) {
  if (rows <= 0) return DFLASH_OK;
  const int64_t warps = rows * heads;
  const unsigned blocks = (unsigned)((warps + 3) / 4);
  Timer t;
  launch_begin(h, DFLASH_K_ELEMENTWISE, s, &t);
  if (dtype == DFLASH_BF16)
    head_norm_rope_kernel<bf16><<<blocks, 128, 0, s>>>(
        in, rows, heads, d, gain, rope ? 1 : 0, rm, len, h->d_rope, h->cfg.max_pos,
        h->cfg.rms_eps, (bf16*)dense, (bf16*)cache, cap, cache_batch, h->d_status);
  else
    head_norm_rope_kernel<float><<<blocks, 128, 0, s>>>(
        in, rows, heads, d, gain, rope ? 1 : 0, rm, len, h->d_rope, h->cfg.max_pos,
        h->cfg.rms_eps, (float*)dense, (float*)cache, cap, cache_batch, h->d_status);
  return launch_end(h, s, &t);
}

int swiglu(dflash_handle* h, cudaStream_t s, int dtype, const float* g, const float* u, void* a,
           int64_t n) {
  if (n <= 0) return DFLASH_OK;
  const unsigned blocks = (unsigned)std::min<int64_t>((n + 255) / 256, 152 * 16);
  Timer t;
  launch_begin(h, DFLASH_K_ELEMENTWISE, s, &t);
  if (dtype == DFLASH_BF16)
    swiglu_kernel<bf16><<<blocks, 256, 0, s>>>(g, u, (bf16*)a, n);
  else
    swiglu_kernel<float><<<blocks, 256, 0, s>>>(g, u, (float*)a, n);
  return launch_end(h, s, &t);
}

int cast_rows(dflash_handle* h, cudaStream_t s, int dtype, const float* in, void* out, int64_t n) {
  if (n <= 0) return DFLASH_OK;
  const unsigned blocks = (unsigned)std::min<int64_t>((n + 255) / 256, 152 * 16);
  Timer t;
  launch_begin(h, DFLASH_K_ELEMENTWISE, s, &t);
  if (dtype == DFLASH_BF16)
    cast_kernel<bf16><<<blocks, 256, 0, s>>>(in, (bf16*)out, n);
  else
    cast_kernel<float><<<blocks, 256, 0, s>>>(in, (float*)out, n);
  return launch_end(h, s, &t);
}

// Bounded-wait self-test: one thread waits, limit_ns at most, on a wait that
// nothing will complete, with the same routines the persistent kernels use —
// which = 0: an mbarrier of this CTA that no thread arrives at; which = 1: a
// device counter that nothing raises (the grid barrier's wait) — and the
// timeout lands in the status word.
__global__ void selftest_wait_kernel(const int* never, int* status, uint64_t limit_ns, int which) {
  __shared__ __align__(8) uint64_t bar;
  if (which == 0) {
    const uint32_t b = ptx::smem_u32(&bar);
    ptx::mbar_init(b, 1);
    ptx::fence_barrier_init();
    if (!ptx::mbar_wait(b, 0, limit_ns)) atomicOr(status, ST_TIMEOUT);
  } else {
    ptx::bounded_wait_geq(never, 1, status, ST_TIMEOUT, limit_ns, 0);
  }
}

int selftest_wait(dflash_handle* h, cudaStream_t s, int which, int64_t limit_ns) {
  Timer t;
  launch_begin(h, DFLASH_K_ELEMENTWISE, s, &t);
  selftest_wait_kernel<<<1, 1, 0, s>>>(h->d_counters + kMaxTiles + 3, h->d_status,
                                       (uint64_t)limit_ns, which);
  return launch_end(h, s, &t);
}

int advance_len(dflash_handle* h, cudaStream_t s, int32_t* len, const int32_t* nrows, int uniform,
                int batch, int cap) {
  Timer t;
  launch_begin(h, DFLASH_K_ELEMENTWISE, s, &t);
  advance_len_kernel<<<(batch + 127) / 128, 128, 0, s>>>(len, nrows, uniform, batch, cap,
                                                         h->d_status);
  return launch_end(h, s, &t);
}

}  // namespace dflash
