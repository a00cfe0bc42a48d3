// Weight-streaming projection for few activation rows (M <= 64).
//
// At draft time every projection multiplies a handful of rows (the B block
// rows of each sequence) by a large bf16 weight, so the work is bound by
// reading the weight once from HBM.  The kernel therefore:
//   * splits the weight into 128-row x 64-column tiles (16 KB) and hands
//     every CTA (one per SM) an equal contiguous run of (tile, k-chunk)
//     units, so all SMs stream the same number of bytes whatever the shape;
//   * stages weight and activation chunks with TMA into an 8-deep
//     shared-memory ring guarded by mbarriers (warp 0 produces, warps 1-8
//     consume: 4 weight-row quarters x 2 k-halves), prefetching the first weight chunks before waiting for the
//     previous kernel (programmatic dependent launch);
//   * multiplies with warp-level bf16 MMA (m16n8k16, fp32 accumulate);
//   * finishes a tile it owns whole with a fused epilogue (fp32 store,
//     residual add, SwiGLU, per-head RMSNorm + RoPE (+ cache append), or
//     per-row top-2 records of an LM-head tile) and writes the partial sums
//     of the (at most two) tiles it shares with neighbours;
//   * after a bounded grid barrier (the grid is co-resident: a cooperative
//     launch of at most two CTAs per SM) gives every (shared tile, row
//     block) to one warp of the grid, which adds the contributors' partials
//     in k order and runs the same epilogue per row;
//   * for the LM head, after a second barrier, merges each row's top-2
//     records over the vocabulary (one warp per row).
#include <string.h>

#include "common.cuh"
#include "ptx.cuh"

namespace dflash {

using namespace ptx;

// Consumer layout: 4 weight-row quarters x WS_KSPLIT slices of each 64-wide
// k-chunk (compile-time tuning), plus one producer warp whose first
// WS_NPROD lanes each issue every WS_NPROD-th stage.
#ifndef DFLASH_WS_KSPLIT
#define DFLASH_WS_KSPLIT 1
#endif
#ifndef DFLASH_WS_NPROD
#define DFLASH_WS_NPROD 1
#endif
constexpr int WS_KSPLIT = DFLASH_WS_KSPLIT;
constexpr int WS_NPROD = DFLASH_WS_NPROD;
static_assert(WS_NPROD == 1, "the producer steps one cursor per lane");
constexpr int WS_CW = 4 * WS_KSPLIT;
constexpr int WS_CT = WS_CW * 32;
constexpr int WS_THREADS = 32 + WS_CT;
constexpr int WS_EPAD = 132;
constexpr int WS_MAXLIST = 1024;   // CTAs per launch at most (one shared tile per CTA boundary)

struct WParams {
  CUtensorMap wmap[WS_MAXMAP];
  CUtensorMap amap[WS_MAXSRC];
  WSeg seg[WS_MAXMAP];
  int nseg, n_tiles, kc, kc_per_src, M, grid, units;
  float* partial;
  int* counters;        // arrival count per tile (last-arriver fix-up)
  int* bar;             // grid barrier word (zero between launches)
  int row_batch;        // rows per reduce task: 4 when tiles have few contributors, else 1
  int* status;
  RowMap rm;
  const int32_t* len;
  const float2* rope_tab;
  int max_pos;
  float eps;
  float4* amx;
  int32_t* ids;
  float* gap;
  int rps_out;
  const int32_t* anchor;
};

static_assert(sizeof(WParams) <= 4096, "kernel parameters must fit the 4 KB limit");

// Ring depth and resident CTAs per SM (compile-time tuning; shared memory per
// CTA must fit 227 KB / WS_MINBLOCKS).
#ifndef DFLASH_WS_STAGES
#define DFLASH_WS_STAGES 8
#endif
// 1: the launch may start while the kernel before it finishes (programmatic
// dependent launch; activations are read after griddepcontrol.wait)
#ifndef DFLASH_WS_PDL
#define DFLASH_WS_PDL 1
#endif
// CTAs per SM.  One, with the deeper ring it leaves room for: with two
// co-resident CTAs a rare result error was seen (one consumer warp's 32
// output columns of one tile, in a few of 300 identical LM-head launches),
// never with one, and one is as fast.  Its cause has not been found, so
// other values are refused.
#ifndef DFLASH_WS_MINBLOCKS
#define DFLASH_WS_MINBLOCKS 1
#endif
static_assert(DFLASH_WS_MINBLOCKS == 1,
              "two streaming CTAs per SM gave rare wrong results whose cause is not located");

template <int MT>
struct WCfg {
  static constexpr int W_BYTES = 128 * 64 * 2;
  static constexpr int A_BYTES = MT * 16 * 64 * 2;
  static constexpr int STAGE_TX = W_BYTES + A_BYTES;
  // deepest ring that fits the shared memory of one of WS_MINBLOCKS CTAs per SM
  static constexpr int BUDGET = DFLASH_WS_MINBLOCKS == 1 ? 232448 : 233472 / DFLASH_WS_MINBLOCKS - 1024;
  static constexpr int FIXED = MT * 16 * WS_EPAD * 4 + 2 * 16 * 8 + 64 + 64 * 8 + 4 * (WS_MAXLIST + 4) + 1024;
  static constexpr int FIT = (BUDGET - FIXED) / STAGE_TX;
  static constexpr int STAGES = FIT < DFLASH_WS_STAGES ? FIT : DFLASH_WS_STAGES;
  static_assert(STAGES >= 2, "ring too shallow");
  static constexpr int OFF_A = STAGES * W_BYTES;
  static constexpr int OFF_E = OFF_A + STAGES * A_BYTES;
  static constexpr int E_FLOATS = MT * 16 * WS_EPAD;
  static constexpr int OFF_BAR = OFF_E + E_FLOATS * 4;
  static constexpr int OFF_MISC = OFF_BAR + 2 * STAGES * 8;
  static constexpr int OFF_LIST = OFF_MISC + 64 + 64 * 8;   // shared tiles, then their count
  static constexpr int SMEM = OFF_LIST + 4 * (WS_MAXLIST + 4) + 1024;
};

__device__ __forceinline__ int seg_of(const WParams& p, int t) {
  int s = 0;
  while (s + 1 < p.nseg && t >= p.seg[s + 1].t0) ++s;
  return s;
}

// CTA that owns unit u when U units are split evenly over G CTAs.
__device__ __forceinline__ int unit_owner(int64_t u, int64_t U, int64_t G) {
  return (int)(((u + 1) * G + U - 1) / U) - 1;
}
__device__ __forceinline__ int first_unit(int64_t c, int64_t U, int64_t G) {
  return (int)(c * U / G);
}

struct Top2 {
  float t1;
  int i1;
  float t2;
};
__device__ __forceinline__ Top2 top2_merge(Top2 a, Top2 b) {
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
__device__ __forceinline__ Top2 top2_warp(Top2 t) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Top2 u;
    u.t1 = __shfl_xor_sync(0xffffffffu, t.t1, o);
    u.i1 = __shfl_xor_sync(0xffffffffu, t.i1, o);
    u.t2 = __shfl_xor_sync(0xffffffffu, t.t2, o);
    t = top2_merge(t, u);
  }
  return t;
}

// ---- epilogues (128 consumer threads, final fp32 tile in E) ------------------
template <int MT>
__device__ void ws_epilogue(const WParams& p, int t, const float* E, volatile int* misc,
                            const int* rowpos) {
  const int tid = threadIdx.x - 32, cw = tid >> 5, lane = threadIdx.x & 31;
  const WSeg& g = p.seg[seg_of(p, t)];
  const int lt = t - g.t0;
  const int M = p.M;
  if (g.kind == SK_F32 || g.kind == SK_RESID) {
    // float4 per thread-iteration; the residual loads of all iterations are
    // issued before any is used (n_valid and ld are multiples of 4 here)
    float* dst = (float*)g.dst;
    constexpr int IT = MT * 512 / WS_CT;  // (MT*16 rows * 32 float4) / consumer threads
    float4 old[IT];
#pragma unroll
    for (int q = 0; q < IT; ++q) {
      const int e = tid + q * WS_CT, r = e >> 5, c = (e & 31) * 4, n = lt * 128 + c;
      old[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (g.kind == SK_RESID && r < M && n < g.n_valid)
        old[q] = *(const float4*)(dst + (int64_t)r * g.ld + n);
    }
#pragma unroll
    for (int q = 0; q < IT; ++q) {
      const int e = tid + q * WS_CT, r = e >> 5, c = (e & 31) * 4, n = lt * 128 + c;
      if (r >= M || n >= g.n_valid) continue;
      const float* ev = E + r * WS_EPAD + c;
      *(float4*)(dst + (int64_t)r * g.ld + n) =
          make_float4(old[q].x + ev[0], old[q].y + ev[1], old[q].z + ev[2], old[q].w + ev[3]);
    }
  } else if (g.kind == SK_SWIGLU) {
    bf16* dst = (bf16*)g.dst;
    for (int e = tid; e < M * 64; e += WS_CT) {
      const int r = e >> 6, c = e & 63;
      const int f = lt * 64 + c;
      if (f >= g.n_valid) continue;
      const float gv = E[r * WS_EPAD + c], uv = E[r * WS_EPAD + 64 + c];
      dst[(int64_t)r * g.ld + f] = __float2bfloat16_rn(gv / (1.0f + expf(-gv)) * uv);
    }
  } else if (g.kind == SK_HEAD) {
    const int d = g.d, half = d >> 1, P = half >> 5, hpt = 128 / d;
    float gn1[2] = {1.f, 1.f}, gn2[2] = {1.f, 1.f};
    if (g.gain != nullptr) {
#pragma unroll
      for (int q = 0; q < 2; ++q)
        if (q < P) {
          gn1[q] = g.gain[lane + 32 * q];
          gn2[q] = g.gain[lane + 32 * q + half];
        }
    }
    for (int pi = cw; pi < M * hpt; pi += WS_CW) {
      const int r = pi / hpt, j = pi - r * hpt;
      const int head = lt * hpt + j;
      const int pb = rowpos[2 * r], pos = rowpos[2 * r + 1];   // sequence, position (-1: skip)
      float2 cs[2] = {make_float2(1.f, 0.f), make_float2(1.f, 0.f)};
      if (g.rope && pos >= 0 && pos < p.max_pos) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (q < P) cs[q] = p.rope_tab[(int64_t)pos * half + lane + 32 * q];
      }
      const float* src = E + r * WS_EPAD + j * d;
      float x1[2], x2[2], ss = 0.f;
#pragma unroll
      for (int q = 0; q < 2; ++q)
        if (q < P) {
          const int jj = lane + 32 * q;
          x1[q] = src[jj];
          x2[q] = src[jj + half];
          ss += x1[q] * x1[q] + x2[q] * x2[q];
        }
      if (g.gain != nullptr) {
        ss = warp_sum(ss);
        const float rinv = 1.0f / sqrtf(ss / (float)d + p.eps);
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (q < P) {
            x1[q] = x1[q] * rinv * gn1[q];
            x2[q] = x2[q] * rinv * gn2[q];
          }
      }
      if (pb < 0) continue;                  // row not appended by this call
      const int b = pb;
      if (g.rope) {
        if (pos < 0 || pos >= p.max_pos) {
          if (lane == 0) atomicOr(p.status, ST_BOUNDS);
          continue;
        }
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (q < P) {
            const float y1 = x1[q] * cs[q].x - x2[q] * cs[q].y;
            const float y2 = x2[q] * cs[q].x + x1[q] * cs[q].y;
            x1[q] = y1;
            x2[q] = y2;
          }
      }
      bf16* o;
      if (g.cache_cap > 0) {
        if (b >= g.cache_batch || pos < 0 || pos >= g.cache_cap) {
          if (lane == 0) atomicOr(p.status, ST_CAPACITY);
          continue;
        }
        o = (bf16*)g.dst + (((int64_t)b * g.cache_heads + head) * g.cache_cap + pos) * d;
      } else {
        o = (bf16*)g.dst + (int64_t)r * g.ld + (int64_t)head * d;
      }
#pragma unroll
      for (int q = 0; q < 2; ++q)
        if (q < P) {
          const int jj = lane + 32 * q;
          o[jj] = __float2bfloat16_rn(x1[q]);
          o[jj + half] = __float2bfloat16_rn(x2[q]);
        }
    }
  } else if (g.kind == SK_ARGMAX) {
    for (int r = cw; r < M; r += WS_CW) {
      Top2 tt{-INFINITY, 0x7fffffff, -INFINITY};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = lane + 32 * q;
        const int n = lt * 128 + c;
        if (n >= g.n_valid) continue;
        const float v = E[r * WS_EPAD + c];
        Top2 u{v, n, -INFINITY};
        tt = top2_merge(tt, u);
      }
      tt = top2_warp(tt);
      if (lane == 0) p.amx[(int64_t)t * M + r] = make_float4(tt.t1, __int_as_float(tt.i1), tt.t2, 0.f);
    }
  }
}

// ---- per-row epilogue of a reduced tile row (one warp, lane = 4 columns) -----
__device__ void ws_row(const WParams& p, int t, int r, float4 v, const int* rowpos) {
  const int lane = threadIdx.x & 31;
  const WSeg& g = p.seg[seg_of(p, t)];
  const int lt = t - g.t0;
  float x[4] = {v.x, v.y, v.z, v.w};
  if (g.kind == SK_F32 || g.kind == SK_RESID) {
    const int n = lt * 128 + 4 * lane;
    if (n < g.n_valid) {   // n_valid and ld are multiples of 4 here
      float4* o = (float4*)((float*)g.dst + (int64_t)r * g.ld + n);
      if (g.kind == SK_RESID) {
        const float4 a = *o;
        x[0] += a.x;
        x[1] += a.y;
        x[2] += a.z;
        x[3] += a.w;
      }
      *o = make_float4(x[0], x[1], x[2], x[3]);
    }
  } else if (g.kind == SK_SWIGLU) {
    // columns 0-63 of the tile are gate rows, 64-127 the matching up rows
    float u[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) u[q] = __shfl_xor_sync(0xffffffffu, x[q], 16);
    if (lane < 16) {
      bf16* dst = (bf16*)g.dst + (int64_t)r * g.ld;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int f = lt * 64 + 4 * lane + q;
        if (f < g.n_valid) dst[f] = __float2bfloat16_rn(x[q] / (1.0f + expf(-x[q])) * u[q]);
      }
    }
  } else if (g.kind == SK_HEAD) {
    // d = 128: one head per tile row; d = 64: two, one per half-warp
    const int d = g.d, half = d >> 1;
    const int hl = d == 128 ? lane : (lane & 15);
    const int head = lt * (128 / d) + (d == 128 ? 0 : (lane >> 4));
    if (g.gain != nullptr) {
      float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
      if (d == 128) ss += __shfl_xor_sync(0xffffffffu, ss, 16);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float rinv = 1.0f / sqrtf(ss / (float)d + p.eps);
#pragma unroll
      for (int q = 0; q < 4; ++q) x[q] = x[q] * rinv * g.gain[4 * hl + q];
    }
    float px[4];   // the element half a head away (the other RoPE operand)
#pragma unroll
    for (int q = 0; q < 4; ++q) px[q] = __shfl_xor_sync(0xffffffffu, x[q], d == 128 ? 16 : 8);
    const int b = rowpos[2 * r], pos = rowpos[2 * r + 1];   // sequence, position (-1: skip)
    if (b < 0) return;                                      // row not appended by this call
    if (g.rope) {
      if (pos < 0 || pos >= p.max_pos) {
        if (lane == 0) atomicOr(p.status, ST_BOUNDS);
        return;
      }
      const bool lo_half = 4 * hl < half;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = (4 * hl + q) - (lo_half ? 0 : half);
        const float2 cs = p.rope_tab[(int64_t)pos * half + i];
        x[q] = lo_half ? x[q] * cs.x - px[q] * cs.y : x[q] * cs.x + px[q] * cs.y;
      }
    }
    bf16* o;
    if (g.cache_cap > 0) {
      if (b >= g.cache_batch || pos < 0 || pos >= g.cache_cap) {
        if (lane == 0) atomicOr(p.status, ST_CAPACITY);
        return;
      }
      o = (bf16*)g.dst + (((int64_t)b * g.cache_heads + head) * g.cache_cap + pos) * d;
    } else {
      o = (bf16*)g.dst + (int64_t)r * g.ld + (int64_t)head * d;
    }
    __nv_bfloat162 t0 = __floats2bfloat162_rn(x[0], x[1]);
    __nv_bfloat162 t1 = __floats2bfloat162_rn(x[2], x[3]);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&t0);
    pk.y = *reinterpret_cast<uint32_t*>(&t1);
    *reinterpret_cast<uint2*>(o + 4 * hl) = pk;
  } else if (g.kind == SK_ARGMAX) {
    Top2 tt{-INFINITY, 0x7fffffff, -INFINITY};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int n = lt * 128 + 4 * lane + q;
      if (n < g.n_valid) tt = top2_merge(tt, Top2{x[q], n, -INFINITY});
    }
    tt = top2_warp(tt);
    if (lane == 0) p.amx[(int64_t)t * p.M + r] = make_float4(tt.t1, __int_as_float(tt.i1), tt.t2, 0.f);
  }
}

// ---- grid barrier (bounded; every CTA of the grid is resident) ---------------
__device__ bool ws_grid_wait(const WParams& p, int target) {
  return bounded_wait_geq(p.bar, target, p.status, ST_TIMEOUT, 2000000000ull, 0);
}
// Consumers of every CTA arrive; true once all CTAs have arrived k times.
// After a timeout (here or in another CTA) the CTA stops taking part.
__device__ bool ws_grid_sync(const WParams& p, int k, volatile int* misc, int tid) {
  named_bar(1, WS_CT);
  if (tid == 0) {
    bool go = misc[0] == 0;
    red_release_gpu_add(p.bar, 1);
    if (go && !ws_grid_wait(p, k * p.grid)) {
      misc[0] = 1;
      go = false;
    }
    misc[4] = go;
  }
  named_bar(1, WS_CT);
  return misc[4] != 0;
}

// ---- shared tiles: one warp per (tile, block of RB rows) over the grid -------
// A tile is shared when a CTA boundary falls strictly inside it (every CTA
// lists these tiles at its start).  Contributor c's partial of tile t is its
// first slot if t is c's first tile, else its second.
template <int MT, int RB>
__device__ void ws_reduce(const WParams& p, const int* rowpos, const int* list) {
  constexpr int CB = 16 / RB;   // contributors whose loads are in flight together
  const int cw = (threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
  const int64_t U = p.units, G = p.grid;
  const int nwarps = p.grid * WS_CW, gw = blockIdx.x * WS_CW + cw;
  const int rblocks = (p.M + RB - 1) / RB;
  const int ntask = list[WS_MAXLIST] * rblocks;
  for (int k = gw; k < ntask; k += nwarps) {
    const int t = list[k / rblocks], r0 = (k - (k / rblocks) * rblocks) * RB;
    const int lo = unit_owner((int64_t)t * p.kc, U, G);
    const int hi = unit_owner((int64_t)t * p.kc + p.kc - 1, U, G);
    float4 sum[RB];
#pragma unroll
    for (int rr = 0; rr < RB; ++rr) sum[rr] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = lo; c0 <= hi; c0 += CB) {
      float4 v[CB][RB];
#pragma unroll
      for (int j = 0; j < CB; ++j) {
        const int cc = min(c0 + j, hi);
        const int slot = 2 * cc + (first_unit(cc, U, G) / p.kc == t ? 0 : 1);
        const float* base = p.partial + (int64_t)slot * (MT * 16 * 128) + 4 * lane;
#pragma unroll
        for (int rr = 0; rr < RB; ++rr)
          v[j][rr] = __ldcg((const float4*)(base + min(r0 + rr, p.M - 1) * 128));
      }
#pragma unroll
      for (int j = 0; j < CB; ++j)
        if (c0 + j <= hi)
#pragma unroll
          for (int rr = 0; rr < RB; ++rr) {
            sum[rr].x += v[j][rr].x;
            sum[rr].y += v[j][rr].y;
            sum[rr].z += v[j][rr].z;
            sum[rr].w += v[j][rr].w;
          }
    }
#pragma unroll
    for (int rr = 0; rr < RB; ++rr)
      if (r0 + rr < p.M) ws_row(p, t, r0 + rr, sum[rr], rowpos);
  }
}

// ---- LM head: each row's top-2 over all vocabulary tiles (one warp per row) --
__device__ void ws_merge(const WParams& p) {
  const int cw = (threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
  const int nwarps = p.grid * WS_CW, gw = blockIdx.x * WS_CW + cw;
  for (int r = gw; r < p.M; r += nwarps) {
    Top2 tt{-INFINITY, 0x7fffffff, -INFINITY};
    for (int t0 = 0; t0 < p.n_tiles; t0 += 32 * 16) {
      float4 rec[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int ti = t0 + lane + 32 * q;
        rec[q] = ti < p.n_tiles ? __ldcg(&p.amx[(int64_t)ti * p.M + r])
                                : make_float4(-INFINITY, __int_as_float(0x7fffffff), -INFINITY, 0.f);
      }
#pragma unroll
      for (int q = 0; q < 16; ++q) tt = top2_merge(tt, Top2{rec[q].x, __float_as_int(rec[q].y), rec[q].z});
    }
    tt = top2_warp(tt);
    if (lane == 0) {
      int64_t out = r, gout = r;
      if (p.rps_out > 0) {
        const int per = p.rps_out - 1;
        const int64_t b = r / per, i = r % per + 1;
        out = b * p.rps_out + i;
        gout = b * per + (i - 1);
        if (i == 1) p.ids[b * p.rps_out] = p.anchor[b];
      }
      float g = tt.t1 - tt.t2;
      p.ids[out] = argmax_id(tt.i1, g, p.status);
      if (p.gap) p.gap[gout] = g;
    }
  }
}

template <int MT, bool GB>
__global__ void __launch_bounds__(WS_THREADS, DFLASH_WS_MINBLOCKS) wstream_kernel(const __grid_constant__ WParams p) {
  using C = WCfg<MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + C::OFF_BAR, bar_empty = bar_full + 8 * C::STAGES;
  volatile int* misc = (volatile int*)(smem + C::OFF_MISC);  // 0 abort, 1 last, 2 issued, 3 consumed
  float* E = (float*)(smem + C::OFF_E);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t U = p.units, G = p.grid;
  const int cta = blockIdx.x;
  const int u0 = first_unit(cta, U, G), u1 = first_unit(cta + 1, U, G);
  const int n = u1 - u0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, WS_CW);
    }
    misc[0] = misc[1] = misc[2] = misc[3] = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) pdl_launch_dependents();

  if (warp == 0) {
    // ---------------- producer: lanes < WS_NPROD issue the TMA loads ---------
    if (lane < WS_NPROD) {
      const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
      // (tile, k-chunk, activation source) of the next unit, stepped without
      // divisions; the tile's weight box is resolved once per tile
      struct Cur {
        int t, kk, src, lk, seg;
        const CUtensorMap* m0;
        const CUtensorMap* m1;   // SwiGLU up half
        int row;
      };
      auto tile = [&](Cur& c) {
        while (c.seg + 1 < p.nseg && c.t >= p.seg[c.seg + 1].t0) ++c.seg;
        const WSeg& g = p.seg[c.seg];
        const int lt = c.t - g.t0;
        c.m0 = &p.wmap[g.map];
        c.m1 = g.kind == SK_SWIGLU ? &p.wmap[g.map2] : nullptr;
        c.row = lt * (g.kind == SK_SWIGLU ? 64 : 128);
      };
      auto start = [&](Cur& c, int u) {
        c.t = u / p.kc;
        c.kk = u - c.t * p.kc;
        c.src = c.kk / p.kc_per_src;
        c.lk = c.kk - c.src * p.kc_per_src;
        c.seg = 0;
        tile(c);
      };
      auto step = [&](Cur& c) {
        if (++c.lk == p.kc_per_src) {
          c.lk = 0;
          ++c.src;
        }
        if (++c.kk == p.kc) {
          c.kk = c.src = c.lk = 0;
          ++c.t;
          tile(c);
        }
      };
      auto issue_w = [&](const Cur& c, int s) {
        const uint32_t dst = sbase + s * C::W_BYTES, bar = bar_full + 8 * s;
        tma_load_2d(dst, c.m0, bar, c.kk * 64, c.row, pol_w);
        if (c.m1 != nullptr) tma_load_2d(dst + C::W_BYTES / 2, c.m1, bar, c.kk * 64, c.row, pol_w);
      };
      auto issue_a = [&](const Cur& c, int s) {
        tma_load_2d(sbase + C::OFF_A + s * C::A_BYTES, &p.amap[c.src], bar_full + 8 * s, c.lk * 64, 0,
                    pol_a);
      };
      Cur wc, ac;
      start(wc, u0);
      ac = wc;
      const int pre = n < C::STAGES ? n : C::STAGES;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(bar_full + 8 * i, C::STAGE_TX);
        issue_w(wc, i);
        step(wc);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i) {
        issue_a(ac, i);
        step(ac);
      }
      int issued = pre;
      // unit i reuses slot i % STAGES after the consumers' release of use
      // i / STAGES - 1, whose phase parity is (i / STAGES - 1) & 1
      int s = pre % C::STAGES;
      uint32_t par = (pre / C::STAGES + 1) & 1;
      for (int i = pre; i < n; ++i) {
        if (misc[0]) break;
        if (!mbar_wait(bar_empty + 8 * s, par)) {
          atomicOr(p.status, ST_TIMEOUT);
          misc[0] = 1;
          break;
        }
        mbar_arrive_expect_tx(bar_full + 8 * s, C::STAGE_TX);
        issue_w(wc, s);
        issue_a(wc, s);
        step(wc);
        issued = i + 1;
        if (++s == C::STAGES) {
          s = 0;
          par ^= 1;
        }
      }
      atomicMax((int*)&misc[2], issued);   // highest stage index issued, for the drain
    }
    __syncwarp();
  } else {
    // ---------------- consumers: warps 1-4, 32 weight rows each -------------
    const int cw = warp - 1, tid = threadIdx.x - 32;
    if (GB && cw == 0) {
      // the shared tiles (a CTA boundary strictly inside), each listed once
      // at its first such boundary; depends on the launch shape only
      int* list = (int*)(smem + C::OFF_LIST);
      int n_shared = 0;
      for (int c0 = 1; c0 < p.grid; c0 += 32) {
        const int c = c0 + lane;
        int t = -1;
        if (c < p.grid) {
          const int fb = first_unit(c, U, G);
          if (fb % p.kc != 0) {
            const int fp = first_unit(c - 1, U, G);
            t = fb / p.kc;
            if (c > 1 && fp % p.kc != 0 && fp / p.kc == t) t = -1;
          }
        }
        const unsigned m = __ballot_sync(0xffffffffu, t >= 0);
        if (t >= 0) list[n_shared + __popc(m & ((1u << lane) - 1u))] = t;
        n_shared += __popc(m);
      }
      if (lane == 0) list[WS_MAXLIST] = n_shared;
    }
    pdl_wait();
    const int nq = cw & 3, kh = cw >> 2;   // weight-row quarter, k-slice of each chunk
    // sequence and cache position of each activation row (head epilogues)
    int* rowpos = (int*)(smem + C::OFF_MISC + 64);
    if (tid < MT * 16) {
      int b = -1, i = 0, pos = -1;
      if (tid < p.M && p.len != nullptr && p.rm.map(tid, b, i)) pos = p.len[b] + i;
      else b = -1;
      rowpos[2 * tid] = b;
      rowpos[2 * tid + 1] = pos;
    }
    named_bar(1, WS_CT);
    float acc[MT][4][4];
    int cur = -1, kbeg = 0, kend = 0, consumed = 0;

    auto flush = [&](int t) {
      named_bar(1, WS_CT);  // the previous epilogue has finished reading E
      const bool full_tile = (kbeg == 0 && kend == p.kc);
      const int g = lane >> 2, tg = lane & 3;
      // the two k-halves of the tile meet in E in a fixed order: half 0 stores,
      // half 1 adds
#pragma unroll
      for (int half = 0; half < WS_KSPLIT; ++half) {
        if (kh == half) {
#pragma unroll
          for (int mb = 0; mb < MT; ++mb)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int col = nq * 32 + j * 8 + 2 * tg;
              float2* e0 = (float2*)&E[(mb * 16 + g) * WS_EPAD + col];
              float2* e1 = (float2*)&E[(mb * 16 + g + 8) * WS_EPAD + col];
              if (half == 0) {
                *e0 = make_float2(acc[mb][j][0], acc[mb][j][1]);
                *e1 = make_float2(acc[mb][j][2], acc[mb][j][3]);
              } else {
                const float2 a0 = *e0, a1 = *e1;
                *e0 = make_float2(a0.x + acc[mb][j][0], a0.y + acc[mb][j][1]);
                *e1 = make_float2(a1.x + acc[mb][j][2], a1.y + acc[mb][j][3]);
              }
            }
        }
        named_bar(1, WS_CT);
      }
      if (!full_tile) {
        // a tile shared with neighbouring CTAs: its partial goes to this
        // CTA's first or second slot
        constexpr int IT = MT * 512 / WS_CT;   // float4s of a tile per consumer thread
        const int first_tile = u0 / p.kc;
        float4* slot = (float4*)(p.partial + (int64_t)(2 * cta + (t == first_tile ? 0 : 1)) * (MT * 16 * 128));
#pragma unroll
        for (int q = 0; q < IT; ++q) {
          const int e4 = tid + q * WS_CT, e = e4 * 4;
          __stcg(slot + e4, *(const float4*)&E[(e >> 7) * WS_EPAD + (e & 127)]);
        }
        if (GB) return;   // finished after the grid barrier
        // otherwise the contributor that arrives last sums the partials in CTA
        // (= k) order, with the loads of up to 8 contributors x all of a
        // thread's float4s issued first, and runs the epilogue
        __threadfence();
        named_bar(1, WS_CT);
        const int lo = unit_owner((int64_t)t * p.kc, U, G);
        const int hi = unit_owner((int64_t)t * p.kc + p.kc - 1, U, G);
        if (tid == 0) {
          const int old = atomicAdd(&p.counters[t], 1);
          const int last = (old == hi - lo);
          if (last) p.counters[t] = 0;
          misc[1] = last;
        }
        named_bar(1, WS_CT);
        if (!misc[1]) return;
        __threadfence();
        float4 sum[IT];
#pragma unroll
        for (int q = 0; q < IT; ++q) sum[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        // CB contributors' partials per batch, all of a thread's float4s of
        // each in flight together (at 64 rows one whole partial per batch:
        // as many dependent batches as contributors, not one per float4);
        // every element still adds the contributors in CTA (= k) order
        constexpr int CB = IT >= 16 ? 2 : IT >= 8 ? 2 : 8;
        for (int c0 = lo; c0 <= hi; c0 += CB) {
          float4 v[CB][IT];
#pragma unroll
          for (int k = 0; k < CB; ++k) {
            const int c = min(c0 + k, hi);
            const int ft = first_unit(c, U, G) / p.kc;
            const float4* src =
                (const float4*)(p.partial + (int64_t)(2 * c + (t == ft ? 0 : 1)) * (MT * 16 * 128));
#pragma unroll
            for (int q = 0; q < IT; ++q) v[k][q] = __ldcg(src + tid + q * WS_CT);
          }
#pragma unroll
          for (int k = 0; k < CB; ++k)
            if (c0 + k <= hi) {
#pragma unroll
              for (int q = 0; q < IT; ++q) {
                sum[q].x += v[k][q].x;
                sum[q].y += v[k][q].y;
                sum[q].z += v[k][q].z;
                sum[q].w += v[k][q].w;
              }
            }
        }
#pragma unroll
        for (int q = 0; q < IT; ++q) {
          const int e = (tid + q * WS_CT) * 4;
          *(float4*)&E[(e >> 7) * WS_EPAD + (e & 127)] = sum[q];
        }
        named_bar(1, WS_CT);
      }
      ws_epilogue<MT>(p, t, E, misc, rowpos);
    };

    // tile / k-chunk of the unit and its ring slot / phase parity, stepped
    // at the top of each turn
    int t = u0 / p.kc, kk = u0 - t * p.kc - 1, s = -1;
    uint32_t fpar = 1;
    for (int i = 0; i < n; ++i) {
      if (++kk == p.kc) {
        kk = 0;
        ++t;
      }
      if (++s == C::STAGES) s = 0;
      if (s == 0) fpar ^= 1;
      if (t != cur) {
        if (cur >= 0) flush(cur);
        cur = t;
        kbeg = kk;
#pragma unroll
        for (int mb = 0; mb < MT; ++mb)
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[mb][j][q] = 0.f;
      }
      kend = kk + 1;
      // after a timed-out wait (in any warp) the warps skip the arithmetic but
      // keep walking the units, so all of them reach the same named barriers
      if (misc[0]) continue;
      // warp-uniform: the phase is complete once any lane has seen it complete
      if (!__any_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, fpar))) {
        if (lane == 0) atomicOr(p.status, ST_TIMEOUT);
        misc[0] = 1;
        continue;
      }
      const uint32_t wb = sbase + s * C::W_BYTES;
      const uint32_t ab = sbase + C::OFF_A + s * C::A_BYTES;
#pragma unroll
      for (int kq = 0; kq < 4 / WS_KSPLIT; ++kq) {
        const int ks = (4 / WS_KSPLIT) * kh + kq;
        uint32_t a[MT][4];
#pragma unroll
        for (int mb = 0; mb < MT; ++mb) {
          const int row = mb * 16 + (lane & 15);
          const int ch = 2 * ks + (lane >> 4);
          ldsm_x4(ab + row * 128 + ((ch ^ (row & 7)) << 4), a[mb][0], a[mb][1], a[mb][2], a[mb][3]);
        }
        uint32_t b[4][2];
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          const int row = nq * 32 + pp * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int ch = 2 * ks + ((lane >> 3) & 1);
          ldsm_x4(wb + row * 128 + ((ch ^ (row & 7)) << 4), b[2 * pp][0], b[2 * pp][1],
                  b[2 * pp + 1][0], b[2 * pp + 1][1]);
        }
#pragma unroll
        for (int mb = 0; mb < MT; ++mb)
#pragma unroll
          for (int j = 0; j < 4; ++j) mma_bf16_16816(acc[mb][j], a[mb], b[j][0], b[j][1]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
      consumed = i + 1;
    }
    if (cur >= 0) flush(cur);
    if (tid == 0) misc[3] = consumed;
    // ---- shared tiles, then (LM head) the vocabulary merge ------------------
    if (GB) {
    const bool argmax = p.seg[0].kind == SK_ARGMAX;
    if (ws_grid_sync(p, 1, misc, tid)) {
      const int* list = (const int*)(smem + C::OFF_LIST);
      if (p.row_batch == 4)
        ws_reduce<MT, 4>(p, rowpos, list);
      else
        ws_reduce<MT, 1>(p, rowpos, list);
    }
    if (argmax && ws_grid_sync(p, 2, misc, tid)) ws_merge(p);
    named_bar(1, WS_CT);
    if (tid == 0) {
      red_release_gpu_add(p.bar, 1);   // this CTA polls the barrier no more
      // once every CTA has left, the first one clears the word for the next launch
      if (blockIdx.x == 0 && !misc[0] && ws_grid_wait(p, (argmax ? 3 : 2) * p.grid)) *p.bar = 0;
    }
    }
  }
  __syncthreads();
  if (misc[0] && threadIdx.x == 0) {
    // drain TMA loads that were issued but never consumed before leaving (at
    // most one ring's worth; each wait is bounded)
    const int hi = min(misc[2], misc[3] + C::STAGES);
    for (int i = misc[3]; i < hi; ++i)
      if (!mbar_wait(bar_full + 8 * (i % C::STAGES), (i / C::STAGES) & 1, 20000000ull)) break;
  }
}

// ---------------------------------------------------------------------------
// GB: the LM head (top-2 records, then a merge over the vocabulary) runs
// with grid barriers and is launched cooperatively; the other projections
// finish shared tiles in the contributor that arrives last.  Both may start
// early (programmatic dependent launch).
template <int MT, bool GB>
static int launch_wstream(dflash_handle* h, cudaStream_t s, int kclass, WParams prm) {
  using C = WCfg<MT>;
  static int occ = -1;
  if (occ < 0) {
    int o = 0;
    if (cudaFuncSetAttribute(wstream_kernel<MT, GB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, wstream_kernel<MT, GB>, WS_THREADS,
                                                      C::SMEM) != cudaSuccess)
      return DFLASH_ERR_CUDA;
    occ = std::min(o, DFLASH_WS_MINBLOCKS);
  }
  if (occ < 1 || (int64_t)occ * h->num_sms > WS_MAXLIST) return DFLASH_ERR_UNSUPPORTED;
  // every CTA resident at once (a grid barrier waits for all of them)
  prm.grid = (int)std::min<int64_t>(prm.units, (int64_t)occ * h->num_sms);
  const int64_t per = prm.units / prm.grid;                 // units of the smallest CTA
  const int64_t contributors = (prm.kc + per - 1) / per + 1;  // at most, per shared tile
  prm.row_batch = contributors <= 4 ? 4 : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.grid);
  cfg.blockDim = dim3(WS_THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (DFLASH_WS_PDL) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na++].val.programmaticStreamSerializationAllowed = 1;
  }
  if (GB) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na++].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  Timer t;
  launch_begin(h, kclass, s, &t);
  cudaLaunchKernelEx(&cfg, wstream_kernel<MT, GB>, prm);
  return launch_end(h, s, &t);
}

size_t wstream_scratch_bytes(const dflash_handle* h, int M) {
  const int mt = (M + 15) / 16;
  return (size_t)2 * h->num_sms * DFLASH_WS_MINBLOCKS * mt * 16 * 128 * sizeof(float) + 256;
}

int wstream(dflash_handle* h, cudaStream_t s, int kclass, const WLaunch& L, float* partial,
            float4* amx) {
  if (L.M < 1 || L.M > 64 || L.K % 64 != 0 || L.nseg < 1 || L.nseg > WS_MAXMAP ||
      L.nsrc < 1 || L.nsrc > WS_MAXSRC || (L.K / 64) % L.nsrc != 0)
    return DFLASH_ERR_SHAPE;
  const int MT = (L.M + 15) / 16;
  WParams prm;
  memset(&prm, 0, sizeof(prm));
  for (int i = 0; i < L.nmap; ++i) prm.wmap[i] = *L.wmaps[i];
  const int kc_per_src = L.K / 64 / L.nsrc;
  for (int i = 0; i < L.nsrc; ++i)
    if (!make_tmap_2d(&prm.amap[i], L.a_src[i], (uint64_t)kc_per_src * 64, (uint64_t)L.M,
                      (uint64_t)L.a_ld * 2, 64, MT * 16))
      return DFLASH_ERR_CUDA;
  for (int i = 0; i < L.nseg; ++i) prm.seg[i] = L.seg[i];
  prm.nseg = L.nseg;
  prm.n_tiles = L.seg[L.nseg - 1].t1;
  prm.kc = L.K / 64;
  prm.kc_per_src = kc_per_src;
  prm.M = L.M;
  prm.units = prm.n_tiles * prm.kc;
  prm.partial = partial;
  prm.counters = h->d_counters;
  prm.bar = h->d_counters + kMaxTiles + 2;
  prm.status = h->d_status;
  prm.rm = L.rm;
  prm.len = L.len;
  prm.rope_tab = h->d_rope;
  prm.max_pos = h->cfg.max_pos;
  prm.eps = h->cfg.rms_eps;
  prm.amx = amx;
  prm.ids = L.ids;
  prm.gap = L.gap;
  prm.rps_out = L.rps_out;
  prm.anchor = L.anchor;
  if (prm.n_tiles > kMaxTiles) return DFLASH_ERR_SHAPE;
  if (L.seg[0].kind == SK_ARGMAX) {
    switch (MT) {
      case 1: return launch_wstream<1, true>(h, s, kclass, prm);
      case 2: return launch_wstream<2, true>(h, s, kclass, prm);
      case 3: return launch_wstream<3, true>(h, s, kclass, prm);
      default: return launch_wstream<4, true>(h, s, kclass, prm);
    }
  }
  switch (MT) {
    case 1: return launch_wstream<1, false>(h, s, kclass, prm);
    case 2: return launch_wstream<2, false>(h, s, kclass, prm);
    case 3: return launch_wstream<3, false>(h, s, kclass, prm);
    default: return launch_wstream<4, false>(h, s, kclass, prm);
  }
}

}  // namespace dflash
