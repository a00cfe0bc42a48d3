// Sampling at temperature T > 0 (txtmix §8): per-row softmax(z / T) with an
// inverse-CDF draw from a given uniform, and the rejection verification of a
// drafted block (accept d_j when u * q(d_j) < p(d_j); at the first rejection
// draw from max(p - q, 0) renormalised, else the bonus from p).
//
// A row of the vocabulary is cut into chunks of SQ_CHUNK indices, one CTA
// per (row, chunk), so a few rows still spread over the whole GPU; each
// thread holds one contiguous slice of SQ_PER indices in registers.  A draw
// follows index order.  Each CTA publishes its chunk's weight; the row's
// last CTA to do so (a fence + counter, no waiting) adds the chunk weights
// in chunk order (one warp: each lane a run of consecutive chunks, then a
// scan across lanes), finds the first chunk whose running end exceeds
// u * total, and records the target's offset in it.  Inside that chunk the
// slices' sums are scanned in thread order and the thread whose slice holds
// the target walks it to the first index whose running sum exceeds it.  An
// index of zero weight is never drawn.  Where rounding leaves the target
// past an interval's end (a target equal to the total, a walk that does not
// cross), the last index of positive weight of that slice, chunk or row is
// taken; a target a rounding error before its chunk's start takes the
// chunk's first index of positive weight: both next to where the draw falls.
//
// All sums are compensated fp32 pairs (hi + lo, about 44 significant bits,
// from error-free two-sum / fma two-product steps): this GPU's fp64 rate is
// a small fraction of its fp32 rate, and fp64 sums, even one thread's,
// dominated the launches.  fp64 remains only in the acceptance test
// u * q(d) < p(d), taken exactly as written.
#include "common.cuh"

namespace dflash {

#ifndef DFLASH_SQ_PER
#define DFLASH_SQ_PER 8
#endif
constexpr int SQ_T = 256, SQ_PER = DFLASH_SQ_PER, SQ_CHUNK = SQ_T * SQ_PER, SQ_STAGE = 1024;
static_assert(SQ_PER % 4 == 0, "slices are whole 16-byte vectors");

static __host__ __device__ __forceinline__ int sq_chunks(int V) {
  return (V + SQ_CHUNK - 1) / SQ_CHUNK;
}

// ---- compensated fp32 arithmetic: value = hi + lo, |lo| <= ulp(hi) / 2 -------------
struct FF {
  float hi, lo;
};
__device__ __forceinline__ FF ff_two_sum(float a, float b) {   // a + b exactly
  const float s = __fadd_rn(a, b), bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ FF ff_renorm(float s, float e) {   // |s| >= |e|
  const float h = __fadd_rn(s, e);
  return {h, __fsub_rn(e, __fsub_rn(h, s))};
}
__device__ __forceinline__ FF ff_add(FF x, FF y) {
  const FF s = ff_two_sum(x.hi, y.hi);
  return ff_renorm(s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo)));
}
__device__ __forceinline__ FF ff_add_f(FF x, float w) {
  const FF s = ff_two_sum(x.hi, w);
  return ff_renorm(s.hi, __fadd_rn(s.lo, x.lo));
}
__device__ __forceinline__ FF ff_neg(FF x) { return {-x.hi, -x.lo}; }
__device__ __forceinline__ FF ff_mul(FF x, FF y) {   // fma two-product of the high parts
  const float p = __fmul_rn(x.hi, y.hi), e = __fmaf_rn(x.hi, y.hi, -p);
  return ff_renorm(p, __fadd_rn(e, __fadd_rn(__fmul_rn(x.hi, y.lo), __fmul_rn(x.lo, y.hi))));
}
__device__ __forceinline__ FF ff_div_f(FF x, float f) {   // f > 0
  const float q1 = __fdiv_rn(x.hi, f);
  const float rem = __fadd_rn(__fmaf_rn(-q1, f, x.hi), x.lo);
  return ff_renorm(q1, __fdiv_rn(rem, f));
}
__device__ __forceinline__ bool ff_lt(FF a, FF b) {
  return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}
__device__ __forceinline__ FF ff_from_d(double u) {
  const float hi = __double2float_rn(u);
  return {hi, __double2float_rn(u - (double)hi)};
}
__device__ __forceinline__ FF ff_shfl(FF x, int src) {
  return {__shfl_sync(0xffffffffu, x.hi, src), __shfl_sync(0xffffffffu, x.lo, src)};
}
__device__ __forceinline__ FF ff_shfl_up(FF x, int o) {
  return {__shfl_up_sync(0xffffffffu, x.hi, o), __shfl_up_sync(0xffffffffu, x.lo, o)};
}
__device__ __forceinline__ FF ff_shfl_xor(FF x, int o) {
  return {__shfl_xor_sync(0xffffffffu, x.hi, o), __shfl_xor_sync(0xffffffffu, x.lo, o)};
}

// Per row (sequence): written by the row's last CTA of the first launch.
struct SqRow {
  FF total;   // the row's total weight (sampling: in units of exp((z - M) / T))
  FF base;    // the target's offset from the owner chunk's start, in the walk's units
  float M;    // sampling: the row's max logit
  float mo;   // sampling: the owner chunk's max logit (the walk's weights are exp((z - mo) / T))
  int owner;  // the chunk that holds the draw (-1: no positive weight)
  int mode;   // verify: 1 = the draw is from p_a (the residual is all zero)
  int a;      // verify: drafts accepted
  int pad;
};

struct SqScratch {
  FF incl[SQ_T];
  FF ffr[SQ_T / 32];
  float fred[SQ_T / 32];
  int ired[SQ_T / 32];
  int pick, a, last;
};

__device__ float sq_block_max(float v, SqScratch* sc) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) sc->fred[wid] = v;
  __syncthreads();
  float m = -INFINITY;
  for (int k = 0; k < SQ_T / 32; ++k) m = fmaxf(m, sc->fred[k]);
  __syncthreads();
  return m;
}

__device__ int sq_block_max_i(int v, SqScratch* sc) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) sc->ired[wid] = v;
  __syncthreads();
  int m = INT_MIN;
  for (int k = 0; k < SQ_T / 32; ++k) m = max(m, sc->ired[k]);
  __syncthreads();
  return m;
}

// The chunk's sum of the threads' values (all threads get it).
__device__ FF sq_block_sum(FF v, SqScratch* sc) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) v = ff_add(v, ff_shfl_xor(v, o));
  if (lane == 0) sc->ffr[wid] = v;
  __syncthreads();
  FF t = sc->ffr[0];
  for (int k = 1; k < SQ_T / 32; ++k) t = ff_add(t, sc->ffr[k]);
  __syncthreads();
  return t;
}

// This thread's slice of chunk c: first index and length (0..SQ_PER).
__device__ __forceinline__ int sq_slice(int c, int V, int& n) {
  const int i0 = min(V, c * SQ_CHUNK + (int)threadIdx.x * SQ_PER);
  n = min(V - i0, SQ_PER);
  return i0;
}

// x[k] = a[i0 + k] for k < n (16-byte loads when the slice is whole and
// aligned).
__device__ __forceinline__ void sq_load(const float* a, int i0, int n, float x[SQ_PER]) {
  const float* s = a + i0;
  if (n == SQ_PER && ((uintptr_t)s & 15) == 0) {
#pragma unroll
    for (int v = 0; v < SQ_PER / 4; ++v) {
      const float4 u = *(const float4*)(s + 4 * v);
      x[4 * v] = u.x, x[4 * v + 1] = u.y, x[4 * v + 2] = u.z, x[4 * v + 3] = u.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < SQ_PER; ++k) x[k] = k < n ? s[k] : 0.f;
  }
}

__device__ __forceinline__ void sq_store(float* a, int i0, int n, const float x[SQ_PER]) {
  float* s = a + i0;
  if (n == SQ_PER && ((uintptr_t)s & 15) == 0) {
#pragma unroll
    for (int v = 0; v < SQ_PER / 4; ++v)
      *(float4*)(s + 4 * v) = make_float4(x[4 * v], x[4 * v + 1], x[4 * v + 2], x[4 * v + 3]);
  } else {
#pragma unroll
    for (int k = 0; k < SQ_PER; ++k)
      if (k < n) s[k] = x[k];
  }
}

// Sum of the slice's weights in index order.
__device__ __forceinline__ FF sq_slice_sum(const float w[SQ_PER], int n) {
  FF s{0.f, 0.f};
#pragma unroll
  for (int k = 0; k < SQ_PER; ++k)
    if (k < n) s = ff_add_f(s, w[k]);
  return s;
}

// exp((x - m) / T) over the slice (0 outside it, and for a chunk of -inf logits).
__device__ __forceinline__ void sq_exp(const float x[SQ_PER], int n, float m, float inv_T,
                                       float w[SQ_PER]) {
#pragma unroll
  for (int k = 0; k < SQ_PER; ++k)
    w[k] = (k < n && m > -INFINITY) ? expf((x[k] - m) * inv_T) : 0.f;
}

// The draw inside the owning chunk, whose slices hold w (all threads call):
// the first index whose running sum from the chunk's start exceeds r.
__device__ int sq_walk(const float w[SQ_PER], int i0, int n, FF r, SqScratch* sc) {
  const int tid = threadIdx.x;
  int first = 0x7fffffff, last = -1;
#pragma unroll
  for (int k = 0; k < SQ_PER; ++k)
    if (k < n && w[k] > 0.f) first = min(first, i0 + k), last = i0 + k;
  if (tid == 0) sc->pick = -1;
  // inclusive scan of the slice sums in thread order (Hillis-Steele)
  sc->incl[tid] = sq_slice_sum(w, n);
  __syncthreads();
  for (int o = 1; o < SQ_T; o <<= 1) {
    const FF add = tid >= o ? sc->incl[tid - o] : FF{0.f, 0.f};
    __syncthreads();
    sc->incl[tid] = ff_add(sc->incl[tid], add);
    __syncthreads();
  }
  const FF lo = tid > 0 ? sc->incl[tid - 1] : FF{0.f, 0.f}, hi = sc->incl[tid];
  if (n > 0 && !ff_lt(r, lo) && ff_lt(r, hi)) {
    FF run = lo;
    int pick = last;   // the walk did not cross: this slice's last positive index
#pragma unroll
    for (int k = 0; k < SQ_PER; ++k) {
      if (k < n) {
        run = ff_add_f(run, w[k]);
        if (ff_lt(r, run)) {
          pick = i0 + k;
          break;
        }
      }
    }
    sc->pick = pick;
  }
  __syncthreads();
  const int found = sc->pick;
  const int lastpos = sq_block_max_i(last, sc);   // r at or past the chunk's end
  const int firstpos = -sq_block_max_i(-first, sc);
  return found >= 0 ? found : (r.hi <= 0.f ? firstpos : lastpos);
}

// Warp 0 of a row's last CTA (lanes in step): the chunk weights v(k) (>= 0)
// added in chunk order, each lane a run of consecutive chunks and a scan
// across the lanes; the owner is the first chunk of positive weight whose
// running end exceeds t = u * total (the last chunk of positive weight when
// none does), pre its running start.  Returns the total.
template <typename Vf>
__device__ FF sq_row_owner(Vf v, int nc, double u, int* owner, FF* pre_owner, FF* t_out) {
  const int lane = threadIdx.x & 31;
  const int g = (nc + 31) / 32, k0 = min(nc, lane * g), k1 = min(nc, k0 + g);
  FF run{0.f, 0.f};
  for (int k = k0; k < k1; ++k) run = ff_add(run, v(k));
  FF incl = run;
  for (int o = 1; o < 32; o <<= 1) {
    const FF y = ff_shfl_up(incl, o);
    if (lane >= o) incl = ff_add(y, incl);
  }
  FF excl = ff_shfl_up(incl, 1);
  if (lane == 0) excl = FF{0.f, 0.f};
  const FF total = ff_shfl(incl, 31);
  const FF t = ff_mul(ff_from_d(u), total);
  FF pre = excl, cpre{0.f, 0.f}, lpre{0.f, 0.f};
  int cand = -1, lastk = -1;
  for (int k = k0; k < k1; ++k) {
    const FF x = v(k);
    const FF end = ff_add(pre, x);
    if (x.hi > 0.f) {
      if (cand < 0 && ff_lt(t, end)) cand = k, cpre = pre;
      lastk = k, lpre = pre;
    }
    pre = end;
  }
  const unsigned bc = __ballot_sync(0xffffffffu, cand >= 0);
  const unsigned bl = __ballot_sync(0xffffffffu, lastk >= 0);
  if (bc) {
    const int src = __ffs(bc) - 1;
    *owner = __shfl_sync(0xffffffffu, cand, src);
    *pre_owner = ff_shfl(cpre, src);
  } else if (bl) {
    const int src = 31 - __clz(bl);
    *owner = __shfl_sync(0xffffffffu, lastk, src);
    *pre_owner = ff_shfl(lpre, src);
  } else {
    *owner = -1;
    *pre_owner = FF{0.f, 0.f};
  }
  *t_out = t;
  return total;
}

// Arrival of this CTA at its row's counter after publishing its chunk's
// record; true in the row's last CTA, which may then read every record.
__device__ bool sq_arrive(int* cnt, int nc, SqScratch* sc) {
  if (threadIdx.x == 0) {
    __threadfence();
    sc->last = atomicAdd(cnt, 1) == nc - 1;
    if (sc->last) {
      *cnt = 0;   // ready for the next call
      __threadfence();
    }
  }
  __syncthreads();
  return sc->last;
}

// A record of the row's chunks: staged in shared memory, or from global
// memory past the stage.
__device__ __forceinline__ float4 sq_rec(const float4* stage, const float4* rec, int k) {
  return k < SQ_STAGE ? stage[k] : __ldcg(rec + k);
}

// ---- per-row softmax and draws ----------------------------------------------------

// (row, chunk): the chunk's max logit m_c and sum of exp((z - m_c) / T),
// record {m_c, sum.hi, sum.lo}; the row's last CTA fills its SqRow (row
// max M, chunk weights sum_c * exp((m_c - M) / T), the owner chunk and the
// target's offset in units of exp((z - m_owner) / T)).
__global__ void __launch_bounds__(SQ_T) sq_stat_kernel(const float* z, int V, int nc, float inv_T,
                                                       const double* __restrict__ u, float4* rec,
                                                       SqRow* rows, int* cnt) {
  __shared__ SqScratch sc;
  __shared__ float4 stage[SQ_STAGE];
  __shared__ float s_f[SQ_STAGE];
  const int64_t row = blockIdx.x / nc;
  const int c = blockIdx.x - (int)(row * nc);
  int n;
  const int i0 = sq_slice(c, V, n);
  float x[SQ_PER], w[SQ_PER];
  sq_load(z + row * V, i0, n, x);
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < SQ_PER; ++k)
    if (k < n) m = fmaxf(m, x[k]);
  m = sq_block_max(m, &sc);
  sq_exp(x, n, m, inv_T, w);
  const FF s = sq_block_sum(sq_slice_sum(w, n), &sc);
  if (threadIdx.x == 0) rec[blockIdx.x] = make_float4(m, s.hi, s.lo, 0.f);
  if (!sq_arrive(cnt + row, nc, &sc)) return;
  const float4* rr = rec + row * nc;
  for (int k = threadIdx.x; k < min(nc, SQ_STAGE); k += SQ_T) stage[k] = __ldcg(rr + k);
  __syncthreads();
  float M = -INFINITY;
  for (int k = threadIdx.x; k < nc; k += SQ_T) M = fmaxf(M, sq_rec(stage, rr, k).x);
  M = sq_block_max(M, &sc);
  // chunk scale factors exp((m_c - M) / T)
  for (int k = threadIdx.x; k < min(nc, SQ_STAGE); k += SQ_T) {
    const float mc = stage[k].x;
    s_f[k] = mc > -INFINITY ? expf((mc - M) * inv_T) : 0.f;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    auto f = [&](int k) {
      if (k < SQ_STAGE) return s_f[k];
      const float mc = __ldcg(rr + k).x;
      return mc > -INFINITY ? expf((mc - M) * inv_T) : 0.f;
    };
    auto vw = [&](int k) {
      const float4 r4 = sq_rec(stage, rr, k);
      return ff_mul(FF{r4.y, r4.z}, FF{f(k), 0.f});
    };
    int owner;
    FF pre, t;
    const FF total = sq_row_owner(vw, nc, u ? u[row] : 0.0, &owner, &pre, &t);
    if (threadIdx.x == 0) {
      SqRow info;
      info.total = total;
      info.M = M;
      info.owner = owner;
      info.mo = owner >= 0 ? sq_rec(stage, rr, owner).x : 0.f;
      FF base = ff_add(t, ff_neg(pre));
      if (base.hi < 0.f) base = FF{0.f, 0.f};
      const float fo = owner >= 0 ? f(owner) : 1.f;
      info.base = fo > 0.f ? ff_div_f(base, fo) : FF{0.f, 0.f};
      info.mode = info.a = info.pad = 0;
      rows[row] = info;
    }
  }
}

// (row, chunk) when probs is given, else one CTA per row at its owner
// chunk: the draw into ids and p = exp((z - M) / T) / total into probs (each
// thread rewrites only its own slice, after reading it, so probs may be z).
__global__ void __launch_bounds__(SQ_T) sq_draw_kernel(const float* z, int V, int nc, int per_row,
                                                       float inv_T, const SqRow* rows,
                                                       int32_t* ids, int skip, float* probs) {
  __shared__ SqScratch sc;
  const int64_t row = blockIdx.x / per_row;
  const SqRow info = rows[row];
  const int c = per_row == 1 ? max(info.owner, 0) : blockIdx.x - (int)(row * per_row);
  int n;
  const int i0 = sq_slice(c, V, n);
  float x[SQ_PER], w[SQ_PER];
  sq_load(z + row * V, i0, n, x);
  if (ids && c == info.owner) {
    sq_exp(x, n, info.mo, inv_T, w);
    const int pick = sq_walk(w, i0, n, info.base, &sc);
    if (threadIdx.x == 0)
      ids[skip > 1 ? row / (skip - 1) * skip + 1 + row % (skip - 1) : row] = pick;
  }
  if (probs) {
    sq_exp(x, n, info.M, inv_T, w);
    const float inv = __fdiv_rn(1.f, info.total.hi);
#pragma unroll
    for (int k = 0; k < SQ_PER; ++k) w[k] = __fmul_rn(w[k], inv);
    sq_store(probs + row * V, i0, n, w);
  }
}

// ---- rejection verification ------------------------------------------------------

// Drafts accepted in sequence b: thread j < B-1 tests d_{j+1} against
// position j (in fp64, as written); a = the first failing j (B-1 when none
// fails).  An id out of range fails its test and sets ST_BOUNDS (from chunk
// 0's CTA).
__device__ int sq_accepted(const int32_t* dr, const float* q, const float* p, int V,
                           const double* u_acc, int B, int64_t b, int c, int* status,
                           SqScratch* sc) {
  if (threadIdx.x == 0) sc->a = B - 1;
  __syncthreads();
  for (int j = threadIdx.x; j < B - 1; j += SQ_T) {
    const int d = dr[j + 1];
    bool ok;
    if (d < 0 || d >= V) {
      ok = false;
      if (c == 0) atomicOr(status, ST_BOUNDS);
    } else {
      const double qd = q[(b * (B - 1) + j) * V + d], pd = p[(b * B + j) * V + d];
      ok = u_acc[b * (B - 1) + j] * qd < pd;
    }
    if (!ok) atomicMin(&sc->a, j);
  }
  __syncthreads();
  return sc->a;
}

// The weights of the draw over this thread's slice: the residual
// max(p_a - q_a, 0) (residual), else p_a itself.
__device__ __forceinline__ void sq_vweights(const float* pa, const float* qa, int i0, int n,
                                            bool residual, float w[SQ_PER]) {
  sq_load(pa, i0, n, w);
  if (residual) {
    float y[SQ_PER];
    sq_load(qa, i0, n, y);
#pragma unroll
    for (int k = 0; k < SQ_PER; ++k) w[k] = fmaxf(__fsub_rn(w[k], y[k]), 0.f);
  }
}

// (sequence, chunk): acceptance; record {residual sum (or p_{B-1} sum after
// full acceptance), p_a sum}; the sequence's last CTA fills its SqRow.
__global__ void __launch_bounds__(SQ_T) sq_vsum_kernel(const int32_t* draft, const float* q,
                                                       const float* p, int V, int nc,
                                                       const double* u_acc,
                                                       const double* __restrict__ u_smp, int B,
                                                       int* status, float4* rec, SqRow* rows,
                                                       int* cnt) {
  __shared__ SqScratch sc;
  __shared__ float4 stage[SQ_STAGE];
  const int64_t b = blockIdx.x / nc;
  const int c = blockIdx.x - (int)(b * nc);
  const int a = sq_accepted(draft + b * B, q, p, V, u_acc, B, b, c, status, &sc);
  const float* pa = p + (b * B + a) * V;
  const float* qa = a < B - 1 ? q + (b * (B - 1) + a) * V : nullptr;
  int n;
  const int i0 = sq_slice(c, V, n);
  float w[SQ_PER];
  sq_vweights(pa, qa, i0, n, a < B - 1, w);
  const FF s = sq_block_sum(sq_slice_sum(w, n), &sc);
  FF sp{0.f, 0.f};
  if (a < B - 1) {
    sq_vweights(pa, qa, i0, n, false, w);
    sp = sq_block_sum(sq_slice_sum(w, n), &sc);
  }
  if (threadIdx.x == 0) rec[blockIdx.x] = make_float4(s.hi, s.lo, sp.hi, sp.lo);
  if (!sq_arrive(cnt + b, nc, &sc)) return;
  const float4* rr = rec + b * nc;
  for (int k = threadIdx.x; k < min(nc, SQ_STAGE); k += SQ_T) stage[k] = __ldcg(rr + k);
  __syncthreads();
  if (threadIdx.x < 32) {
    // mode 1 when the residual is all zero (p_a == q_a): the draw is from p_a
    int any = 0;
    for (int k = threadIdx.x; k < nc; k += 32) any |= sq_rec(stage, rr, k).x > 0.f;
    const int mode = (a < B - 1 && !__any_sync(0xffffffffu, any)) ? 1 : 0;
    auto vw = [&](int k) {
      const float4 r4 = sq_rec(stage, rr, k);
      return mode ? FF{r4.z, r4.w} : FF{r4.x, r4.y};
    };
    int owner;
    FF pre, t;
    const FF total = sq_row_owner(vw, nc, u_smp[b], &owner, &pre, &t);
    if (threadIdx.x == 0) {
      SqRow info;
      info.total = total;
      FF base = ff_add(t, ff_neg(pre));
      if (base.hi < 0.f) base = FF{0.f, 0.f};
      info.base = base;
      info.M = info.mo = 0.f;
      info.owner = owner;
      info.mode = mode;
      info.a = a;
      info.pad = 0;
      rows[b] = info;
    }
  }
}

// One CTA per sequence: the token after the accepted prefix (a walk of the
// owner chunk) and the sequence's outputs.
__global__ void __launch_bounds__(SQ_T) sq_vdraw_kernel(
    const int32_t* draft, const float* q, const float* p, int V, int B, const int32_t* start,
    const SqRow* rows, int32_t* accept, int32_t* tau, int32_t* token, int32_t* out_tokens,
    int32_t* new_len) {
  __shared__ SqScratch sc;
  const int64_t b = blockIdx.x;
  const SqRow info = rows[b];
  const int a = info.a;
  const float* pa = p + (b * B + a) * V;
  const float* qa = a < B - 1 ? q + (b * (B - 1) + a) * V : nullptr;
  int n;
  const int i0 = sq_slice(max(info.owner, 0), V, n);
  float w[SQ_PER];
  sq_vweights(pa, qa, i0, n, a < B - 1 && info.mode == 0, w);
  const int tok = info.owner >= 0 ? sq_walk(w, i0, n, info.base, &sc) : -1;
  if (threadIdx.x == 0) {
    const int32_t* dr = draft + b * B;
    int32_t* out = out_tokens + b * B;
    for (int j = 0; j < B; ++j) out[j] = j < a ? dr[j + 1] : (j == a ? tok : -1);
    accept[b] = a;
    if (tau) tau[b] = a + 1;
    if (token) token[b] = tok;
    if (new_len) new_len[b] = start[b] + a + 1;
  }
}

// Scratch: [rows * nc] chunk records (16 bytes), [rows] SqRow, [rows] counters.
size_t sampling_ws_bytes(int rows, int V) {
  return (size_t)rows * ((size_t)sq_chunks(V) * 16 + 48) + 512;
}

struct SqWs {
  float4* rec;
  SqRow* rows;
  int* cnt;
};
static SqWs carve_sq(void* ws, int rows, int nc) {
  char* p = (char*)ws;
  SqWs o;
  o.rec = (float4*)p;
  p += (size_t)rows * nc * 16;
  o.rows = (SqRow*)p;
  p += (size_t)rows * sizeof(SqRow);
  o.cnt = (int*)p;
  return o;
}
static_assert(sizeof(SqRow) + sizeof(int) <= 48, "per-row scratch");

int sample_rows(dflash_handle* h, cudaStream_t s, const float* logits, int rows, int V, float T,
                const double* u, int32_t* ids, int ids_skip_first_of, float* probs, void* ws) {
  const int nc = sq_chunks(V);
  const int64_t units = (int64_t)rows * nc;
  if (units > 0x7fffffff) return DFLASH_ERR_INVALID_ARG;
  const SqWs w = carve_sq(ws, rows, nc);
  const float inv_T = 1.0f / T;
  const int per_row = probs ? nc : 1;
  if (cudaMemsetAsync(w.cnt, 0, (size_t)rows * sizeof(int), s) != cudaSuccess)
    return DFLASH_ERR_CUDA;
  Timer t;
  launch_begin(h, DFLASH_K_LM_HEAD, s, &t);
  sq_stat_kernel<<<(unsigned)units, SQ_T, 0, s>>>(logits, V, nc, inv_T, ids ? u : nullptr, w.rec,
                                                  w.rows, w.cnt);
  sq_draw_kernel<<<(unsigned)((int64_t)rows * per_row), SQ_T, 0, s>>>(
      logits, V, nc, per_row, inv_T, w.rows, ids, ids_skip_first_of, probs);
  count_launch();   // two kernels: launch_end counts one
  return launch_end(h, s, &t);
}

int verify_rejection(dflash_handle* h, cudaStream_t s, const int32_t* draft, const float* q,
                     const float* p, int V, const double* u_acc, const double* u_smp, int batch,
                     int B, const int32_t* start, int32_t* accept, int32_t* tau, int32_t* token,
                     int32_t* out_tokens, int32_t* new_len, void* ws) {
  const int nc = sq_chunks(V);
  const int64_t units = (int64_t)batch * nc;
  if (units > 0x7fffffff) return DFLASH_ERR_INVALID_ARG;
  const SqWs w = carve_sq(ws, batch, nc);
  if (cudaMemsetAsync(w.cnt, 0, (size_t)batch * sizeof(int), s) != cudaSuccess)
    return DFLASH_ERR_CUDA;
  Timer t;
  launch_begin(h, DFLASH_K_VERIFY, s, &t);
  sq_vsum_kernel<<<(unsigned)units, SQ_T, 0, s>>>(draft, q, p, V, nc, u_acc, u_smp, B,
                                                  h->d_status, w.rec, w.rows, w.cnt);
  sq_vdraw_kernel<<<batch, SQ_T, 0, s>>>(draft, q, p, V, B, start, w.rows, accept, tau, token,
                                         out_tokens, new_len);
  count_launch();   // two kernels: launch_end counts one
  return launch_end(h, s, &t);
}

}  // namespace dflash
