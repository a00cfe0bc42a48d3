// DFlash 2 candidate selection (txtmix source reading §13-§14), greedy: each
// draft position keeps its top-K tokens by logit; starting from the anchor,
// a walk picks at every position the candidate b maximising
//   S_t(a, b) = U_t(b) + <A(a) * H_t, Bc(b)>,   H_t = W_h xhat_t,
// a the token picked before it (xhat_t the final-normed hidden row).
//
// The walk is serial only in which predecessor it follows, so the pair term
// is computed for every (candidate of position t-1, candidate of position
// t) pair in parallel first; the walk then reads K-entry score rows.
//
// Launches: (1) one CTA per (row, chunk of SL_CHUNK vocabulary entries):
// the chunk's best entry; (2) one warp per row: tau, the K-th best chunk
// maximum, and the chunks kept by it (a chunk whose best entry ranks after
// tau cannot hold any of the row's top K); (3) one CTA per kept chunk: its
// top K; (4) one CTA per row: the kept lists sorted (bitonic, whole CTA),
// the first K are the row's candidates and their logits; (5) the gate before its norm, W_h (x * g),
// and the rows' sums of squares, tiled (32 gate entries x 16 rows x a split
// of the hidden axis) so that each W_h entry is read once per 16 rows;
// (6) one CTA per position row: H_t (the splits added, scaled by 1 / rms)
// and the row's K x K table of pair scores plus U_t; (7) one CTA per
// sequence: the walk over its tables.  Each step reads what the launch
// before it wrote, so no CTA waits on or counts another.
//
// Order: a ranks before b when a's value is larger, or equal with the lower
// id; top-K lists are in that order and a score tie keeps the earlier
// candidate.  A warp's top K over its lanes' entries is bounded by the K-th
// best of the lanes' best entries: the few entries ranked at or before it
// are gathered one per lane and sorted across the warp (bitonic); when more
// than 32 are, each lane sorts its own entries and K rounds take the best
// head.
#include "common.cuh"

namespace dflash {

constexpr int SL_T = 256, SL_PER = 8, SL_CHUNK = SL_T * SL_PER;
constexpr int SL_RS = 32;        // rank slice of one pair-score CTA

static __host__ __device__ __forceinline__ int sl_chunks(int V) {
  return (V + SL_CHUNK - 1) / SL_CHUNK;
}

__device__ __forceinline__ bool sl_before(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

// Sort a lane's E entries into rank order (odd-even transposition network,
// static indices, so the entries stay in registers).
template <int E>
__device__ __forceinline__ void sl_sort(float (&v)[E], int (&id)[E]) {
#pragma unroll
  for (int pass = 0; pass < E; ++pass) {
#pragma unroll
    for (int k = pass & 1; k + 1 < E; k += 2) {
      if (sl_before(v[k + 1], id[k + 1], v[k], id[k])) {
        const float tv = v[k];
        const int ti = id[k];
        v[k] = v[k + 1], id[k] = id[k + 1];
        v[k + 1] = tv, id[k + 1] = ti;
      }
    }
  }
}

// One (v, id) per lane sorted across the warp into rank order (bitonic;
// lane 0 ends with the best).
__device__ __forceinline__ void sl_warp_sort(float& v, int& id) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, j);
      const int oi = __shfl_xor_sync(0xffffffffu, id, j);
      // the lower lane of a pair keeps the better entry in runs sorted best
      // first (bit k of the lane clear), the worse one in the other runs
      const bool keep_better = ((lane & j) == 0) == ((lane & k) == 0 || k == 32);
      const bool take = keep_better ? sl_before(ov, oi, v, id) : sl_before(v, id, ov, oi);
      if (take) v = ov, id = oi;
    }
  }
}

// The warp's top K over its lanes' E entries each (v, id), in rank order,
// into out_v / out_id.  Padding entries are (-inf, INT_MAX); real ids are
// distinct.  The K-th best of the lanes' best entries, tau, bounds the
// answer: only entries ranked at or before tau can be in it, and at least K
// are.  When at most 32 are, they are gathered one per lane (through the
// warp's 32-entry scratch) and sorted across the warp; otherwise each lane
// sorts its entries and K rounds take the best head.
template <int E>
__device__ void sl_warp_topk(float (&v)[E], int (&id)[E], int K, float* out_v, int* out_id,
                             float* sv, int* si) {
  const int lane = threadIdx.x & 31;
  float mv = v[0];
  int mi = id[0];
#pragma unroll
  for (int e = 1; e < E; ++e)
    if (sl_before(v[e], id[e], mv, mi)) mv = v[e], mi = id[e];
  sl_warp_sort(mv, mi);
  const float tv = __shfl_sync(0xffffffffu, mv, K - 1);
  const int ti = __shfl_sync(0xffffffffu, mi, K - 1);
  int cnt = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) cnt += !sl_before(tv, ti, v[e], id[e]);
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  if (total <= 32) {
    int pos = incl - cnt;
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (!sl_before(tv, ti, v[e], id[e])) sv[pos] = v[e], si[pos] = id[e], ++pos;
    __syncwarp();
    float cv = lane < total ? sv[lane] : -INFINITY;
    int ci = lane < total ? si[lane] : INT_MAX;
    __syncwarp();
    sl_warp_sort(cv, ci);
    if (lane < K) out_v[lane] = cv, out_id[lane] = ci;
    return;
  }
  sl_sort(v, id);
  for (int r = 0; r < K; ++r) {
    float bv = v[0];
    int bid = id[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bid, o);
      if (sl_before(ov, oi, bv, bid)) bv = ov, bid = oi;
    }
    if (lane == 0) out_v[r] = bv, out_id[r] = bid;
    if (id[0] == bid && v[0] == bv) {   // this lane's head was taken (or both are padding)
#pragma unroll
      for (int e = 0; e + 1 < E; ++e) v[e] = v[e + 1], id[e] = id[e + 1];
      v[E - 1] = -INFINITY, id[E - 1] = INT_MAX;
    }
  }
}

struct SlTopScratch {
  float v[SL_T / 32][DFLASH_SEL_KMAX];
  int id[SL_T / 32][DFLASH_SEL_KMAX];
  float gv[SL_T / 32][32];   // each warp's gathering scratch
  int gi[SL_T / 32][32];
  int last;
};

// The CTA's top K from the 8 warps' lists in sc (warp 0 calls): lane l holds
// entries l, l + 32, ... of the 8K concatenated entries.
__device__ void sl_merge_warps(SlTopScratch* sc, int K, float* out_v, int* out_id) {
  const int lane = threadIdx.x & 31;
  float v[8];
  int id[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int e = lane + 32 * m, w = e / DFLASH_SEL_KMAX, k = e % DFLASH_SEL_KMAX;
    const bool ok = w < SL_T / 32 && k < K;
    v[m] = ok ? sc->v[w][k] : -INFINITY;
    id[m] = ok ? sc->id[w][k] : INT_MAX;
  }
  sl_warp_topk(v, id, K, out_v, out_id, sc->gv[0], sc->gi[0]);
}

// The slice of chunk c this thread holds: 8 entries (v, id), padding past V.
__device__ __forceinline__ void sl_load_slice(const float* z, int V, int c, float (&v)[SL_PER],
                                              int (&id)[SL_PER]) {
  const int i0 = c * SL_CHUNK + (int)threadIdx.x * SL_PER;
  if (i0 + SL_PER <= V && ((uintptr_t)(z + i0) & 15) == 0) {
    const float4 a = *(const float4*)(z + i0), b = *(const float4*)(z + i0 + 4);
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
#pragma unroll
    for (int k = 0; k < SL_PER; ++k) id[k] = i0 + k;
  } else {
#pragma unroll
    for (int k = 0; k < SL_PER; ++k) {
      const int i = i0 + k;
      v[k] = i < V ? z[i] : -INFINITY;
      id[k] = i < V ? i : INT_MAX;
    }
  }
}

// Launch 1: (row, chunk): the chunk's best entry into cm_v / cm_i [rows][nc].
__global__ void __launch_bounds__(SL_T) sl_cmax_kernel(const float* __restrict__ logits, int V,
                                                       int nc, float* cm_v, int* cm_i) {
  __shared__ float wv[SL_T / 32];
  __shared__ int wi[SL_T / 32];
  const int64_t row = blockIdx.x / nc;
  const int c = blockIdx.x - (int)(row * nc);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  float v[SL_PER];
  int id[SL_PER];
  sl_load_slice(logits + row * V, V, c, v, id);
  float bv = v[0];
  int bi = id[0];
#pragma unroll
  for (int k = 1; k < SL_PER; ++k)
    if (sl_before(v[k], id[k], bv, bi)) bv = v[k], bi = id[k];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (sl_before(ov, oi, bv, bi)) bv = ov, bi = oi;
  }
  if (lane == 0) wv[wid] = bv, wi[wid] = bi;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < SL_T / 32; ++w)
      if (sl_before(wv[w], wi[w], bv, bi)) bv = wv[w], bi = wi[w];
    cm_v[blockIdx.x] = bv, cm_i[blockIdx.x] = bi;
  }
}

// Warp 0: tau, the K-th best of the row's nc (<= 256) chunk maxima, into
// sc->tv / sc->ti (padding when nc < K, which keeps every chunk).  The row's
// top K all rank at or before tau: K chunks have a best entry at or before
// it.  So a chunk whose best entry ranks after tau holds none of them.
struct SlTau {
  float lv[DFLASH_SEL_KMAX];
  int li[DFLASH_SEL_KMAX];
  float gv[32];
  int gi[32];
  float tv;
  int ti;
};
__device__ void sl_row_tau(const float* cm_v, const int* cm_i, int nc, int K, SlTau* t) {
  const int lane = threadIdx.x & 31;
  float v[8];
  int id[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int c = lane + 32 * m;
    v[m] = c < nc ? cm_v[c] : -INFINITY;
    id[m] = c < nc ? cm_i[c] : INT_MAX;
  }
  sl_warp_topk(v, id, K, t->lv, t->li, t->gv, t->gi);
  __syncwarp();
  if (lane == 0) t->tv = t->lv[K - 1], t->ti = t->li[K - 1];
}

// Launch 2: one warp per row: tau and the row's kept chunks (best entry
// ranked at or before tau), in chunk order, into kept [rows][256] and
// nkept [rows].
__global__ void __launch_bounds__(SL_T) sl_tau_kernel(const float* cm_v, const int* cm_i,
                                                      int rows, int nc, int K, int* kept,
                                                      int* nkept) {
  __shared__ SlTau tau[SL_T / 32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t row = (int64_t)blockIdx.x * (SL_T / 32) + wid;
  if (row >= rows) return;
  SlTau* t = &tau[wid];
  const float* rv = cm_v + row * nc;
  const int* ri = cm_i + row * nc;
  sl_row_tau(rv, ri, nc, K, t);
  __syncwarp();
  int base = 0;
  for (int c0 = 0; c0 < nc; c0 += 32) {
    const int c = c0 + lane;
    const bool keep = c < nc && !sl_before(t->tv, t->ti, rv[c], ri[c]);
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (keep) kept[row * 256 + base + __popc(m & ((1u << lane) - 1))] = c;
    base += __popc(m);
  }
  if (lane == 0) nkept[row] = base;
}

// Launch 3: (row, slot): the top K of the row's kept chunk in that slot into
// rec_v / rec_i [rows][nc][K] (by slot); slots past nkept exit at once.
__global__ void __launch_bounds__(SL_T) sl_topk_kernel(const float* __restrict__ logits, int V,
                                                       int nc, int K, const int* kept,
                                                       const int* nkept, float* rec_v,
                                                       int* rec_i) {
  __shared__ SlTopScratch sc;
  const int64_t row = blockIdx.x / nc;
  const int slot = blockIdx.x - (int)(row * nc);
  if (slot >= nkept[row]) return;
  const int c = kept[row * 256 + slot];
  const int wid = threadIdx.x >> 5;
  float v[SL_PER];
  int id[SL_PER];
  sl_load_slice(logits + row * V, V, c, v, id);
  sl_warp_topk(v, id, K, sc.v[wid], sc.id[wid], sc.gv[wid], sc.gi[wid]);
  __syncthreads();
  const int64_t rbase = ((int64_t)row * nc + slot) * K;
  if (wid == 0) sl_merge_warps(&sc, K, rec_v + rbase, rec_i + rbase);
}

// Launch 4: one CTA per row: the kept chunks' lists (nkept * K entries,
// padded to a power of two) sorted into rank order in shared memory by the
// whole CTA (bitonic; runs with bit k of the index clear are sorted best
// first, the others worst first), and the first K into cand / unary.
constexpr int SL_MERGE_MAX = 4096;   // 256 chunks x DFLASH_SEL_KMAX
__global__ void __launch_bounds__(SL_T) sl_merge_kernel(const float* rec_v, const int* rec_i,
                                                        const int* nkept, int nc, int K,
                                                        int32_t* cand, float* unary) {
  __shared__ float ev[SL_MERGE_MAX];
  __shared__ int ei[SL_MERGE_MAX];
  const int64_t row = blockIdx.x;
  const int tid = threadIdx.x;
  const int n = nkept[row] * K;
  int P = 2;
  while (P < n) P <<= 1;
  for (int e = tid; e < P; e += SL_T) {
    const bool ok = e < n;
    ev[e] = ok ? rec_v[row * nc * K + e] : -INFINITY;
    ei[e] = ok ? rec_i[row * nc * K + e] : INT_MAX;
  }
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int t = tid; t < P / 2; t += SL_T) {
        const int a = 2 * t - (t & (j - 1)), c = a + j;
        const bool best_first = (a & k) == 0;
        const bool swap = best_first ? sl_before(ev[c], ei[c], ev[a], ei[a])
                                     : sl_before(ev[a], ei[a], ev[c], ei[c]);
        if (swap) {
          const float tv = ev[a];
          const int ti = ei[a];
          ev[a] = ev[c], ei[a] = ei[c];
          ev[c] = tv, ei[c] = ti;
        }
      }
      __syncthreads();
    }
  }
  if (tid < K) unary[row * K + tid] = ev[tid], cand[row * K + tid] = ei[tid];
}

struct SlPairArgs {
  const float* x;       // [batch * B, D] residual stream after the last layer
  const float* gain;    // [D] final RMSNorm gain
  const int32_t* anchor;
  const void* w_h;      // [rank, D]
  const void* code_pred, *code_succ;   // [n_codes, rank]
  const int32_t* cand;  // [rows][K]
  const float* unary;   // [rows][K]
  float* gpart;         // [KZ][rows][rank] partial W_h (x * g) over the K splits
  float* gssq;          // [KZ][rows] partial sums of x^2
  float* part;          // [rows][K][K] the walk's tables
  int32_t* draft_ids;   // [batch, B]
  float* scores;        // [batch, B - 1] (nullable)
  int* status;
  float eps;
  int B, D, rank, K, n_codes, S, KZ, rows;
};

template <typename T>
__device__ __forceinline__ float sl_ld(const void* p, int64_t i) {
  return to_f(((const T*)p)[i]);
}

constexpr int SG_ROWS = 16, SG_KT = 64, SG_SPLIT = 256;

// 8 consecutive weights as floats (one 16-byte load for bf16, two for fp32).
__device__ __forceinline__ void sl_ld8(const bf16* p, float w[8]) {
  const uint4 u = *(const uint4*)p;
  const uint32_t a[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    w[2 * k] = __uint_as_float(a[k] << 16);
    w[2 * k + 1] = __uint_as_float(a[k] & 0xffff0000u);
  }
}
__device__ __forceinline__ void sl_ld8(const float* p, float w[8]) {
  const float4 u = *(const float4*)p, v = *(const float4*)(p + 4);
  w[0] = u.x, w[1] = u.y, w[2] = u.z, w[3] = u.w, w[4] = v.x, w[5] = v.y, w[6] = v.z, w[7] = v.w;
}

// The context gate before its norm, W_h (x * g), and the rows' sums of
// squares, as partial sums over K splits of SG_SPLIT entries.  CTA (slice
// s, group of SG_ROWS position rows, split kz): a 32 x SG_ROWS tile of
// outputs; W_h (one 16-byte load per thread and tile) and x * g (one) are
// staged through shared memory SG_KT entries at a time, so every W_h entry
// is read once per row group.  D is a multiple of SG_KT and the rows are
// 16-byte aligned (checked by the caller).  The pair kernel adds the splits
// in split order and scales by 1 / rms.
template <typename T>
__global__ void __launch_bounds__(SL_T) sl_gate_kernel(SlPairArgs P) {
  __shared__ float Ws[SL_RS][SG_KT + 1];
  __shared__ float Xs[SG_ROWS][SG_KT + 1];
  const int tid = threadIdx.x, nb = P.B - 1;
  const int ngroups = (P.rows + SG_ROWS - 1) / SG_ROWS;
  const int s = blockIdx.x % P.S, gi = (blockIdx.x / P.S) % ngroups,
            kz = blockIdx.x / (P.S * ngroups);
  const int r0 = gi * SG_ROWS, d_lo = kz * SG_SPLIT, d_hi = min(P.D, d_lo + SG_SPLIT);
  const int orow = tid / 16, oc = (tid % 16) * 2;   // this thread's output row and column pair
  const int wr = tid / 8, wc = (tid % 8) * 8;       // its W_h tile entries
  const int xr = tid / 16, xc = (tid % 16) * 4;     // its x tile entries
  const int pr_x = r0 + xr;
  const float* xrow = nullptr;
  if (pr_x < P.rows) {
    const int64_t b = pr_x / nb, t = pr_x - b * nb;
    xrow = P.x + (b * P.B + 1 + t) * P.D;
  }
  const T* wrow = (const T*)P.w_h + (int64_t)(s * SL_RS + wr) * P.D;
  float acc0 = 0.f, acc1 = 0.f, ssq = 0.f;
  // the next tile's entries are loaded into registers while this one is used
  float w8[8];
  float4 xn = make_float4(0.f, 0.f, 0.f, 0.f), gn = xn;
  sl_ld8(wrow + d_lo + wc, w8);
  if (xrow) xn = *(const float4*)(xrow + d_lo + xc), gn = *(const float4*)(P.gain + d_lo + xc);
  for (int d0 = d_lo; d0 < d_hi; d0 += SG_KT) {
#pragma unroll
    for (int k = 0; k < 8; ++k) Ws[wr][wc + k] = w8[k];
    float4 xv = xn;
    ssq = fmaf(xv.x, xv.x, fmaf(xv.y, xv.y, fmaf(xv.z, xv.z, fmaf(xv.w, xv.w, ssq))));
    xv = make_float4(xv.x * gn.x, xv.y * gn.y, xv.z * gn.z, xv.w * gn.w);
    Xs[xr][xc] = xv.x, Xs[xr][xc + 1] = xv.y, Xs[xr][xc + 2] = xv.z, Xs[xr][xc + 3] = xv.w;
    __syncthreads();
    if (d0 + SG_KT < d_hi) {
      sl_ld8(wrow + d0 + SG_KT + wc, w8);
      if (xrow)
        xn = *(const float4*)(xrow + d0 + SG_KT + xc), gn = *(const float4*)(P.gain + d0 + SG_KT + xc);
    }
#pragma unroll 8
    for (int dd = 0; dd < SG_KT; ++dd) {
      const float xs = Xs[orow][dd];
      acc0 = fmaf(Ws[oc][dd], xs, acc0);
      acc1 = fmaf(Ws[oc + 1][dd], xs, acc1);
    }
    __syncthreads();
  }
  const int pr = r0 + orow;
  if (pr < P.rows) {
    float* g = P.gpart + ((int64_t)kz * P.rows + pr) * P.rank + s * SL_RS + oc;
    g[0] = acc0;
    g[1] = acc1;
  }
  if (s == 0) {   // row xr's sum of squares over the split: its 16 threads are a half-warp
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
    if ((tid % 16) == 0 && pr_x < P.rows) P.gssq[(int64_t)kz * P.rows + pr_x] = ssq;
  }
}

constexpr int SL_RMAX = 1024;   // largest rank

// Launch 4: one CTA per position row.  H_t = (the gate's splits added) /
// rms; the gated predecessor rows A(a) * H_t (a: the anchor at t = 0, else
// position t-1's candidates) and the successor rows Bc(c) gathered once
// into shared memory (rows padded by one word against bank conflicts); the
// K x K table U_t(c_j) + <A(a_i) * H_t, Bc(c_j)> written out.
template <typename T>
__global__ void __launch_bounds__(SL_T) sl_table_kernel(SlPairArgs P) {
  extern __shared__ float dyn[];
  __shared__ float Hs[SL_RMAX];
  const int tid = threadIdx.x;
  const int nb = P.B - 1, K = P.K, rank = P.rank, Rp = rank + 1;
  const int64_t pr = blockIdx.x, b = pr / nb;
  const int t = (int)(pr - b * nb);
  __shared__ int ids_p[DFLASH_SEL_KMAX], ids_s[DFLASH_SEL_KMAX];
  const int npred = t == 0 ? 1 : K;
  if (tid < K) {
    int a = 0;
    if (tid < npred) {
      a = t == 0 ? P.anchor[b] : P.cand[(pr - 1) * K + tid];
      if (a < 0 || a >= P.n_codes) {
        atomicOr(P.status, ST_BOUNDS);
        a = 0;
      }
    }
    ids_p[tid] = a;
    ids_s[tid] = P.cand[pr * K + tid];
  }
  // the splits added in split order (up to 8 loads in flight), scaled by 1 / rms
  float ss = 0.f;
#pragma unroll 8
  for (int kz = 0; kz < P.KZ; ++kz) ss += P.gssq[(int64_t)kz * P.rows + pr];
  const float rinv = 1.0f / sqrtf(ss / (float)P.D + P.eps);
  for (int r = tid; r < rank; r += SL_T) {
    float hv = 0.f;
#pragma unroll 8
    for (int kz = 0; kz < P.KZ; ++kz) hv += P.gpart[((int64_t)kz * P.rows + pr) * rank + r];
    Hs[r] = hv * rinv;
  }
  __syncthreads();
  float* Ag = dyn;            // [K][Rp]
  float* Bg = dyn + K * Rp;   // [K][Rp]
  constexpr int U = 8;        // gathers in flight per thread
  for (int e0 = tid; e0 < K * rank; e0 += SL_T * U) {
    float av[U], bv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = e0 + u * SL_T, i = e / rank, r = e - i * rank;
      av[u] = bv[u] = 0.f;
      if (e < K * rank) {
        if (i < npred) av[u] = sl_ld<T>(P.code_pred, (int64_t)ids_p[i] * rank + r);
        bv[u] = sl_ld<T>(P.code_succ, (int64_t)ids_s[i] * rank + r);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = e0 + u * SL_T, i = e / rank, r = e - i * rank;
      if (e < K * rank) {
        Ag[i * Rp + r] = av[u] * Hs[r];
        Bg[i * Rp + r] = bv[u];
      }
    }
  }
  __syncthreads();
  float* tab = P.part + pr * K * K;
  for (int e = tid; e < K * K; e += SL_T) {
    const int i = e / K, j = e - i * K;
    const float* ar = Ag + i * Rp;
    const float* br = Bg + j * Rp;
    float acc = 0.f;
#pragma unroll 8
    for (int r = 0; r < rank; ++r) acc = fmaf(ar[r], br[r], acc);
    tab[e] = P.unary[pr * K + j] + acc;
  }
}

// Launch 5: one CTA per sequence: its tables (nb K K scores) and
// candidates (nb K ids) into shared memory, then warp 0 walks them from the
// anchor.
__global__ void __launch_bounds__(SL_T) sl_walk_kernel(SlPairArgs P) {
  extern __shared__ float dyn[];
  const int tid = threadIdx.x, lane = tid & 31;
  const int nb = P.B - 1, K = P.K;
  const int64_t b = blockIdx.x;
  int* ci = (int*)(dyn + nb * K * K);
  for (int e = tid; e < nb * K * K; e += SL_T) dyn[e] = P.part[b * nb * K * K + e];
  for (int e = tid; e < nb * K; e += SL_T) ci[e] = P.cand[b * nb * K + e];
  __syncthreads();
  if (tid >= 32) return;
  int pi = 0;   // the predecessor's candidate index (the anchor's row at t = 0)
  for (int tt = 0; tt < nb; ++tt) {
    float sc = -INFINITY;
    int j = INT_MAX;
    if (lane < K) sc = dyn[(tt * K + pi) * K + lane], j = lane;
    for (int o = 16; o > 0; o >>= 1) {
      const float os = __shfl_xor_sync(0xffffffffu, sc, o);
      const int oj = __shfl_xor_sync(0xffffffffu, j, o);
      if (sl_before(os, oj, sc, j)) sc = os, j = oj;
    }
    if (lane == 0) {
      P.draft_ids[b * P.B + 1 + tt] = ci[tt * K + j];
      if (P.scores) P.scores[b * nb + tt] = sc;
    }
    pi = j;
  }
  if (lane == 0) P.draft_ids[b * P.B] = P.anchor[b];
}

// Scratch: chunk maxima [rows][nc] and lists [rows][nc][K] (value, id), candidates and logits
// [rows][K], gate partials [KZ][rows][rank] and [KZ][rows], the walk's
// tables [rows][K][K].
struct SlWs {
  float* cm_v;
  int* cm_i;
  int* kept;
  int* nkept;
  float* rec_v;
  int* rec_i;
  int32_t* cand;
  float* unary;
  float* gpart;
  float* gssq;
  float* part;
};
static int sl_splits(int D) { return (D + SG_SPLIT - 1) / SG_SPLIT; }
static SlWs carve_sl(void* ws, int rows, int nc, int K, int rank, int KZ) {
  auto up = [](size_t n) { return (n + 255) & ~(size_t)255; };
  char* p = (char*)ws;
  SlWs o;
  const size_t lists = (size_t)rows * nc * K;
  o.cm_v = (float*)p, p += up((size_t)rows * nc * 4);
  o.cm_i = (int*)p, p += up((size_t)rows * nc * 4);
  o.kept = (int*)p, p += up((size_t)rows * 256 * 4);
  o.nkept = (int*)p, p += up((size_t)rows * 4);
  o.rec_v = (float*)p, p += up(lists * 4);
  o.rec_i = (int*)p, p += up(lists * 4);
  o.cand = (int32_t*)p, p += up((size_t)rows * K * 4);
  o.unary = (float*)p, p += up((size_t)rows * K * 4);
  o.gpart = (float*)p, p += up((size_t)KZ * rows * rank * 4);
  o.gssq = (float*)p, p += up((size_t)KZ * rows * 4);
  o.part = (float*)p;
  return o;
}

size_t select_ws_bytes(int batch, int B, int V, int D, int K, int rank) {
  const size_t rows = (size_t)batch * (B - 1), nc = sl_chunks(V), KZ = sl_splits(D);
  return rows * nc * (K + 1) * 8 + rows * 257 * 4 + rows * K * 8 + KZ * rows * (rank + 1) * 4 +
         rows * K * K * 4 + 12 * 256;
}

static size_t sl_table_smem(int K, int rank) { return (size_t)2 * K * (rank + 1) * sizeof(float); }
static size_t sl_walk_smem(int B, int K) { return (size_t)(B - 1) * K * (K + 1) * sizeof(float); }

// Checked by the caller: 1 <= K <= min(DFLASH_SEL_KMAX, V); rank a multiple
// of SL_RS, at most SL_RMAX; D a multiple of SG_KT; nc <= 256;
// nc K <= SL_MERGE_MAX; the table and walk kernels' shared memory within 200 KB.
bool select_shape_ok(int B, int V, int D, int K, int rank) {
  const int nc = sl_chunks(V);
  return B >= 2 && D % SG_KT == 0 && nc <= 256 && K >= 1 && K <= DFLASH_SEL_KMAX && K <= V &&
         rank >= SL_RS && rank % SL_RS == 0 && rank <= SL_RMAX &&
         nc * K <= SL_MERGE_MAX && sl_table_smem(K, rank) <= 200 * 1024 &&
         sl_walk_smem(B, K) <= 200 * 1024;
}

template <typename T>
static void sl_launch_table(const SlPairArgs& P, unsigned grid, size_t smem, cudaStream_t s) {
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(sl_table_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
  sl_table_kernel<T><<<grid, SL_T, smem, s>>>(P);
}

int select_candidates(dflash_handle* h, cudaStream_t s, const float* logits, const float* x,
                      const float* gain, const int32_t* anchor, int batch, int B, int K,
                      const void* w_h, int rank, const void* code_pred, const void* code_succ,
                      int n_codes, int32_t* draft_ids, int32_t* cand_out, float* scores,
                      void* ws) {
  const dflash_config& cf = h->cfg;
  const int V = cf.vocab, D = cf.hidden, rows = batch * (B - 1), nc = sl_chunks(V);
  const int S = rank / SL_RS, KZ = sl_splits(D), ngroups = (rows + SG_ROWS - 1) / SG_ROWS;
  if ((int64_t)rows * nc > 0x7fffffff) return DFLASH_ERR_INVALID_ARG;
  SlWs w = carve_sl(ws, rows, nc, K, rank, KZ);
  if (cand_out) w.cand = cand_out;
  SlPairArgs P;
  P.x = x, P.gain = gain, P.anchor = anchor, P.w_h = w_h, P.code_pred = code_pred;
  P.code_succ = code_succ, P.cand = w.cand, P.unary = w.unary, P.gpart = w.gpart;
  P.gssq = w.gssq, P.part = w.part, P.draft_ids = draft_ids;
  P.scores = scores, P.status = h->d_status, P.eps = cf.rms_eps, P.B = B, P.D = D;
  P.rank = rank, P.K = K, P.n_codes = n_codes, P.S = S, P.KZ = KZ, P.rows = rows;
  const unsigned gate_grid = (unsigned)(S * ngroups * KZ);
  const size_t wsm = sl_walk_smem(B, K);
  if (wsm > 48 * 1024)
    cudaFuncSetAttribute(sl_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wsm);
  Timer t;
  launch_begin(h, DFLASH_K_LM_HEAD, s, &t);
  const unsigned units = (unsigned)((int64_t)rows * nc);
  sl_cmax_kernel<<<units, SL_T, 0, s>>>(logits, V, nc, w.cm_v, w.cm_i);
  sl_tau_kernel<<<(unsigned)((rows + 7) / 8), SL_T, 0, s>>>(w.cm_v, w.cm_i, rows, nc, K, w.kept,
                                                            w.nkept);
  sl_topk_kernel<<<units, SL_T, 0, s>>>(logits, V, nc, K, w.kept, w.nkept, w.rec_v, w.rec_i);
  sl_merge_kernel<<<(unsigned)rows, SL_T, 0, s>>>(w.rec_v, w.rec_i, w.nkept, nc, K, w.cand,
                                                  w.unary);
  if (cf.dtype == DFLASH_BF16) {
    sl_gate_kernel<bf16><<<gate_grid, SL_T, 0, s>>>(P);
    sl_launch_table<bf16>(P, (unsigned)rows, sl_table_smem(K, rank), s);
  } else {
    sl_gate_kernel<float><<<gate_grid, SL_T, 0, s>>>(P);
    sl_launch_table<float>(P, (unsigned)rows, sl_table_smem(K, rank), s);
  }
  sl_walk_kernel<<<(unsigned)batch, SL_T, wsm, s>>>(P);
  for (int k = 0; k < 6; ++k) count_launch();   // seven kernels: launch_end counts one
  return launch_end(h, s, &t);
}

}  // namespace dflash
