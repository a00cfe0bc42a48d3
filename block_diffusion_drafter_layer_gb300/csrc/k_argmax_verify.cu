// Integer-deciding kernels: row argmax over fp32 logits (lowest index on
// ties, top-1 minus top-2 gap) and greedy block verification.
#include "common.cuh"

namespace dflash {

struct Top2 {
  float t1;
  int i1;
  float t2;
};

// Merge two partial (top1, index, top2) summaries; ties keep the lower index.
__device__ __forceinline__ Top2 merge_top2(Top2 a, Top2 b) {
  Top2 r;
  if (b.t1 > a.t1 || (b.t1 == a.t1 && b.i1 < a.i1)) {
    r.t1 = b.t1;
    r.i1 = b.i1;
  } else {
    r.t1 = a.t1;
    r.i1 = a.i1;
  }
  r.t2 = fmaxf(fminf(a.t1, b.t1), fmaxf(a.t2, b.t2));
  return r;
}

__global__ void __launch_bounds__(256) argmax_rows_kernel(const float* __restrict__ logits, int V,
                                                          int32_t* ids, float* gap, int rps_out,
                                                          const int32_t* anchor, int* status) {
  __shared__ Top2 part[8];
  const int64_t r = blockIdx.x;
  const float* z = logits + r * V;
  Top2 t{-INFINITY, 0x7fffffff, -INFINITY};
  for (int j = threadIdx.x; j < V; j += blockDim.x) {
    const float v = z[j];
    if (v > t.t1) {
      t.t2 = t.t1;
      t.t1 = v;
      t.i1 = j;
    } else if (v > t.t2) {
      t.t2 = v;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Top2 u;
    u.t1 = __shfl_xor_sync(0xffffffffu, t.t1, o);
    u.i1 = __shfl_xor_sync(0xffffffffu, t.i1, o);
    u.t2 = __shfl_xor_sync(0xffffffffu, t.t2, o);
    t = merge_top2(t, u);
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) part[wid] = t;
  __syncthreads();
  if (threadIdx.x == 0) {
    Top2 a = part[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) a = merge_top2(a, part[w]);
    int64_t out = r, gout = r;
    if (rps_out > 0) {
      const int per = rps_out - 1;
      const int64_t b = r / per, i = r % per + 1;
      out = b * rps_out + i;
      gout = b * per + (i - 1);
      if (i == 1) ids[b * rps_out] = anchor[b];
    }
    float g = a.t1 - a.t2;
    ids[out] = argmax_id(a.i1, g, status);
    if (gap) gap[gout] = g;
  }
}

int argmax_rows(dflash_handle* h, cudaStream_t s, const float* logits, int64_t rows, int V,
                int32_t* ids, float* gap, int rows_per_seq_out, const int32_t* anchor) {
  if (rows <= 0) return DFLASH_OK;
  Timer t;
  launch_begin(h, DFLASH_K_LM_HEAD, s, &t);
  argmax_rows_kernel<<<(unsigned)rows, 256, 0, s>>>(logits, V, ids, gap, rows_per_seq_out, anchor,
                                                    h->d_status);
  return launch_end(h, s, &t);
}

// Greedy verification, one thread per sequence (txtmix §8): the accepted
// length is the number of leading draft positions that equal the target's
// argmax at the previous position; the bonus is the target's argmax right
// after the accepted prefix.
__global__ void verify_greedy_kernel(const int32_t* __restrict__ draft,
                                     const int32_t* __restrict__ post, int batch, int B,
                                     const int32_t* start, int32_t* accept, int32_t* tau,
                                     int32_t* bonus, int32_t* out_tokens, int32_t* new_len) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int32_t* dr = draft + (int64_t)b * B;
  const int32_t* po = post + (int64_t)b * B;
  int a = 0;
  while (a < B - 1 && dr[a + 1] == po[a]) ++a;
  const int32_t bon = po[a];
  int32_t* out = out_tokens + (int64_t)b * B;
  for (int j = 0; j < B; ++j) out[j] = (j < a) ? dr[j + 1] : (j == a ? bon : -1);
  const int32_t st = start[b];
  accept[b] = a;
  bonus[b] = bon;
  if (tau) tau[b] = a + 1;
  if (new_len) new_len[b] = st + a + 1;
}

int verify_greedy(cudaStream_t s, const int32_t* draft, const int32_t* post, int batch, int B,
                  const int32_t* start, int32_t* accept, int32_t* tau, int32_t* bonus,
                  int32_t* out_tokens, int32_t* new_len) {
  verify_greedy_kernel<<<(batch + 127) / 128, 128, 0, s>>>(draft, post, batch, B, start, accept,
                                                           tau, bonus, out_tokens, new_len);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

// Device-side bookkeeping of a round (one thread per sequence): the round's
// emitted tokens (the accepted drafts and the bonus, tau[b] of them) are
// appended to the sequence's output at out_len[b], and tau is logged, so a
// loop of rounds needs no host read in between.  A tau outside [1, B] flags
// ST_BOUNDS and emits nothing; tokens past out_cap are counted, not stored.
__global__ void emit_tokens_kernel(const int32_t* __restrict__ out_tokens,
                                   const int32_t* __restrict__ tau, int batch, int B,
                                   int32_t* out_buf, int out_cap, int32_t* out_len,
                                   int32_t* tau_log, int log_cap, int32_t* n_rounds,
                                   int* status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int n = tau[b];
  if (n < 1 || n > B) {
    atomicOr(status, ST_BOUNDS);
    return;
  }
  const int at = out_len[b];
  for (int j = 0; j < n; ++j)
    if (at + j < out_cap) out_buf[(int64_t)b * out_cap + at + j] = out_tokens[(int64_t)b * B + j];
  out_len[b] = at + n;
  if (tau_log && n_rounds) {
    const int r = n_rounds[b];
    if (r < log_cap) tau_log[(int64_t)b * log_cap + r] = n;
    n_rounds[b] = r + 1;
  }
}

int emit_tokens(cudaStream_t s, const int32_t* out_tokens, const int32_t* tau, int batch, int B,
                int32_t* out_buf, int out_cap, int32_t* out_len, int32_t* tau_log, int log_cap,
                int32_t* n_rounds, int* status) {
  emit_tokens_kernel<<<(batch + 127) / 128, 128, 0, s>>>(out_tokens, tau, batch, B, out_buf, out_cap,
                                                         out_len, tau_log, log_cap, n_rounds, status);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

}  // namespace dflash
