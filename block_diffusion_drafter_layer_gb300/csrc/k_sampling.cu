// Sampling at temperature T > 0 (txtmix §8): per-row softmax(z / T) with an
// inverse-CDF draw from a given uniform, and the rejection verification of a
// drafted block (accept d_j when u * q(d_j) < p(d_j); at the first rejection
// draw from max(p - q, 0) renormalised, else the bonus from p).
//
// A draw follows the vocabulary's index order: each of the CTA's threads owns
// one contiguous slice, sums its weights in fp64 in order, the slice sums are
// scanned in thread order, and the thread whose slice holds u * total walks
// it in order to the first index whose running sum exceeds u * total.  An
// index of zero weight is never drawn.
#include "common.cuh"

namespace dflash {

constexpr int SP_THREADS = 1024;

struct DrawScratch {
  double sum[SP_THREADS];
  int last[SP_THREADS / 32];
  int found;
  float fmax[SP_THREADS / 32];
};

// Smallest index i with running sum of w(0..i) > u * total (all threads
// call; the CTA's threads are SP_THREADS).  Returns the index and the total.
template <typename Wf>
__device__ int draw_index(Wf w, int V, double u, DrawScratch* sc, double* total_out) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int per = (V + SP_THREADS - 1) / SP_THREADS;
  const int i0 = min(V, tid * per), i1 = min(V, i0 + per);
  double s = 0.0;
  int last = -1;
  for (int i = i0; i < i1; ++i) {
    const float x = w(i);
    s += (double)x;
    if (x > 0.f) last = i;
  }
  // inclusive scan of the slice sums in thread order (Hillis-Steele)
  sc->sum[tid] = s;
  for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  if (lane == 0) sc->last[wid] = last;
  if (tid == 0) sc->found = -1;
  __syncthreads();
  for (int o = 1; o < SP_THREADS; o <<= 1) {
    const double add = tid >= o ? sc->sum[tid - o] : 0.0;
    __syncthreads();
    sc->sum[tid] += add;
    __syncthreads();
  }
  const double total = sc->sum[SP_THREADS - 1];
  const double t = u * total;
  const double lo = tid > 0 ? sc->sum[tid - 1] : 0.0;
  if (i0 < i1 && lo <= t && t < sc->sum[tid]) {
    double run = lo;
    int pick = -1;
    for (int i = i0; i < i1; ++i) {
      run += (double)w(i);
      if (run > t) {
        pick = i;
        break;
      }
    }
    if (pick >= 0) sc->found = pick;
  }
  __syncthreads();
  int r = sc->found;
  if (r < 0) {   // u * total rounded up to the total: the last index of positive weight
    r = -1;
    for (int k = 0; k < SP_THREADS / 32; ++k) r = max(r, sc->last[k]);
  }
  __syncthreads();   // the scratch may be reused right after
  if (total_out) *total_out = total;
  return r;
}

__device__ float block_max_f(float v, DrawScratch* sc) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) sc->fmax[wid] = v;
  __syncthreads();
  float m = -INFINITY;
  for (int k = 0; k < SP_THREADS / 32; ++k) m = fmaxf(m, sc->fmax[k]);
  __syncthreads();
  return m;
}

// One CTA per row: p = softmax(z / T) (fp32 exponentials, fp64 sums); the
// row's draw with u[row] into ids[row * ids_stride] (when ids is given) and
// p into probs[row] (when probs is given).
__global__ void __launch_bounds__(SP_THREADS) sample_rows_kernel(const float* __restrict__ logits,
                                                                 int V, float inv_T,
                                                                 const double* __restrict__ u,
                                                                 int32_t* ids, int ids_stride,
                                                                 float* probs) {
  __shared__ DrawScratch sc;
  const int64_t row = blockIdx.x;
  const float* z = logits + row * V;
  float m = -INFINITY;
  for (int i = threadIdx.x; i < V; i += SP_THREADS) m = fmaxf(m, z[i]);
  m = block_max_f(m, &sc);
  auto w = [&](int i) { return expf((z[i] - m) * inv_T); };
  double total = 0.0;
  const int pick = draw_index(w, V, u ? u[row] : 0.0, &sc, &total);
  if (ids && threadIdx.x == 0) ids[row * ids_stride] = pick;
  if (probs) {
    const float inv = (float)(1.0 / total);
    for (int i = threadIdx.x; i < V; i += SP_THREADS) probs[row * V + i] = w(i) * inv;
  }
}

// One CTA per sequence.  q: [batch, B-1, V] the drafts' distributions; p:
// [batch, B, V] the target's; u_acc: [batch, B-1]; u_smp: [batch].
__global__ void __launch_bounds__(SP_THREADS) verify_rejection_kernel(
    const int32_t* __restrict__ draft, const float* __restrict__ q, const float* __restrict__ p,
    int V, const double* __restrict__ u_acc, const double* __restrict__ u_smp, int B,
    const int32_t* start, int32_t* accept, int32_t* tau, int32_t* token, int32_t* out_tokens,
    int32_t* new_len, int* status) {
  __shared__ DrawScratch sc;
  __shared__ int s_a;
  const int64_t b = blockIdx.x;
  const int32_t* dr = draft + b * B;
  if (threadIdx.x == 0) {
    int a = 0;
    while (a < B - 1) {
      const int d = dr[a + 1];
      if (d < 0 || d >= V) {
        atomicOr(status, ST_BOUNDS);
        break;
      }
      const double qd = q[(b * (B - 1) + a) * V + d], pd = p[(b * B + a) * V + d];
      if (u_acc[b * (B - 1) + a] * qd < pd) ++a;
      else break;
    }
    s_a = a;
  }
  __syncthreads();
  const int a = s_a;
  const float* pa = p + (b * B + a) * V;
  int tok;
  if (a < B - 1) {
    const float* qa = q + (b * (B - 1) + a) * V;
    double total = 0.0;
    tok = draw_index([&](int i) { return fmaxf(pa[i] - qa[i], 0.f); }, V, u_smp[b], &sc, &total);
    if (!(total > 0.0)) tok = draw_index([&](int i) { return pa[i]; }, V, u_smp[b], &sc, nullptr);
  } else {
    tok = draw_index([&](int i) { return pa[i]; }, V, u_smp[b], &sc, nullptr);
  }
  if (threadIdx.x == 0) {
    int32_t* out = out_tokens + b * B;
    for (int j = 0; j < B; ++j) out[j] = j < a ? dr[j + 1] : (j == a ? tok : -1);
    accept[b] = a;
    if (tau) tau[b] = a + 1;
    if (token) token[b] = tok;
    if (new_len) new_len[b] = start[b] + a + 1;
  }
}

int sample_rows(dflash_handle* h, cudaStream_t s, const float* logits, int rows, int V, float T,
                const double* u, int32_t* ids, int ids_stride, float* probs) {
  Timer t;
  launch_begin(h, DFLASH_K_LM_HEAD, s, &t);
  sample_rows_kernel<<<rows, SP_THREADS, 0, s>>>(logits, V, 1.0f / T, u, ids, ids_stride, probs);
  return launch_end(h, s, &t);
}

int verify_rejection(dflash_handle* h, cudaStream_t s, const int32_t* draft, const float* q,
                     const float* p, int V, const double* u_acc, const double* u_smp, int batch,
                     int B, const int32_t* start, int32_t* accept, int32_t* tau, int32_t* token,
                     int32_t* out_tokens, int32_t* new_len) {
  Timer t;
  launch_begin(h, DFLASH_K_VERIFY, s, &t);
  verify_rejection_kernel<<<batch, SP_THREADS, 0, s>>>(draft, q, p, V, u_acc, u_smp, B, start,
                                                       accept, tau, token, out_tokens, new_len,
                                                       h->d_status);
  return launch_end(h, s, &t);
}

}  // namespace dflash
