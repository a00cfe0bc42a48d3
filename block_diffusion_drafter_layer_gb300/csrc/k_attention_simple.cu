// Reference-schedule attention kernel: one CTA per (block row, query head).
// Scores for every visible key go to shared memory, then max, exp, sum and
// the value average run in fixed key order.  Keys are the sequence's cached
// context followed by the block's own rows (draft: bidirectional unless the
// layer is causal or windowed, txtmix §6), or the cache up to the row's own
// position (causal target).
#include "common.cuh"

namespace dflash {

template <typename T>
__global__ void __launch_bounds__(256) attention_simple_kernel(
    const T* __restrict__ q, const T* __restrict__ kc, const T* __restrict__ vc, int cap,
    const int32_t* __restrict__ len, const T* __restrict__ kb, const T* __restrict__ vb, int rps,
    int H, int G, int d, int causal_in_cache, T* __restrict__ o, float scale, int max_keys,
    int* status, int causal, int window) {
  extern __shared__ float sm[];
  __shared__ float red[33];
  float* qs = sm;
  float* sc = sm + d;
  const int r = blockIdx.x, hq = blockIdx.y;
  const int b = r / rps, i = r - b * rps;
  const int g = hq / (H / G);
  const int L = len[b];
  int nctx, nblk;
  if (causal_in_cache) {
    nctx = L + i + 1;
    nblk = 0;
  } else {
    nctx = L;
    nblk = rps;
  }
  const int nk = nctx + nblk;
  T* orow = o + (int64_t)r * (H * d) + (int64_t)hq * d;
  if (nk > max_keys || nctx > cap || L < 0) {
    if (threadIdx.x == 0) atomicOr(status, ST_BOUNDS);
    for (int k = threadIdx.x; k < d; k += blockDim.x) orow[k] = from_f<T>(0.f);
    return;
  }
  const T* qrow = q + (int64_t)r * (H * d) + (int64_t)hq * d;
  for (int k = threadIdx.x; k < d; k += blockDim.x) qs[k] = to_f(qrow[k]);
  __syncthreads();
  const T* kcb = kc + ((int64_t)b * G + g) * cap * d;
  const T* vcb = vc + ((int64_t)b * G + g) * cap * d;
  const T* kbb = kb ? kb + (int64_t)b * rps * (G * d) + (int64_t)g * d : nullptr;
  const T* vbb = vb ? vb + (int64_t)b * rps * (G * d) + (int64_t)g * d : nullptr;
  // the draft row's visible keys [k0, k1): causal up to its own position
  // L + i, a window the last `window` positions (the row itself always)
  int k0 = 0, k1 = nk;
  if (!causal_in_cache) {
    if (causal) k1 = L + i + 1;
    if (window > 0) k0 = max(0, L + i - window + 1);
  }

  float mloc = -INFINITY;
  for (int j = k0 + threadIdx.x; j < k1; j += blockDim.x) {
    const T* kr = (j < nctx) ? kcb + (int64_t)j * d : kbb + (int64_t)(j - nctx) * (G * d);
    float s = 0.f;
    for (int k = 0; k < d; ++k) s = fmaf(qs[k], to_f(kr[k]), s);
    s *= scale;
    sc[j] = s;
    mloc = fmaxf(mloc, s);
  }
  const float m = block_max(mloc, red);
  float lloc = 0.f;
  for (int j = k0 + threadIdx.x; j < k1; j += blockDim.x) {
    const float p = expf(sc[j] - m);
    sc[j] = p;
    lloc += p;
  }
  const float l = block_sum(lloc, red);   // ends with a barrier: sc[] is complete
  for (int k = threadIdx.x; k < d; k += blockDim.x) {
    float acc = 0.f;
    for (int j = k0; j < k1; ++j) {
      const T* vr = (j < nctx) ? vcb + (int64_t)j * d : vbb + (int64_t)(j - nctx) * (G * d);
      acc = fmaf(sc[j], to_f(vr[k]), acc);
    }
    orow[k] = from_f<T>(acc / l);
  }
}

int attention(dflash_handle* h, cudaStream_t s, int dtype, const void* q, const void* kc,
              const void* vc, int cap, const int32_t* len, const void* kb, const void* vb,
              int batch, int rows_per_seq, int H, int G, int d, bool causal_in_cache, void* o,
              int causal, int window) {
  const int max_keys = cap + (causal_in_cache ? 0 : rows_per_seq);
  const size_t smem = (size_t)(d + max_keys) * sizeof(float);
  if (smem > 227 * 1024) return DFLASH_ERR_SHAPE;
  const float scale = 1.0f / sqrtf((float)d);
  const dim3 grid(batch * rows_per_seq, H);
  Timer t;
  launch_begin(h, DFLASH_K_ATTENTION, s, &t);
  if (dtype == DFLASH_BF16) {
    cudaFuncSetAttribute(attention_simple_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    attention_simple_kernel<bf16><<<grid, 256, smem, s>>>(
        (const bf16*)q, (const bf16*)kc, (const bf16*)vc, cap, len, (const bf16*)kb,
        (const bf16*)vb, rows_per_seq, H, G, d, causal_in_cache ? 1 : 0, (bf16*)o, scale, max_keys,
        h->d_status, causal, window);
  } else {
    cudaFuncSetAttribute(attention_simple_kernel<float>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attention_simple_kernel<float><<<grid, 256, smem, s>>>(
        (const float*)q, (const float*)kc, (const float*)vc, cap, len, (const float*)kb,
        (const float*)vb, rows_per_seq, H, G, d, causal_in_cache ? 1 : 0, (float*)o, scale,
        max_keys, h->d_status, causal, window);
  }
  return launch_end(h, s, &t);
}

}  // namespace dflash
