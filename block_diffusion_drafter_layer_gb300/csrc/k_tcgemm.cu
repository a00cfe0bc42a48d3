// Dense projection on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Used where a projection multiplies many rows (the context prefill: fusing
// and injecting thousands of target positions at once), so the work is a
// dense contraction.  One CTA per SM walks 128-row x BN-column output tiles
// (BN = 256, or 128 where 256-column tiles would leave most SMs idle):
//   warp 0    one lane streams 64-wide K slices of the activations (A, 16 KB)
//             and of the weight (B, BN x 128 B) with TMA into a 4-deep
//             (BN = 256) or 6-deep (BN = 128) ring;
//   warp 1    allocates two BN-column TMEM accumulators; one lane issues
//             tcgen05.mma (M=128, N=BN, K=16, bf16 in, fp32 accumulate) into
//             the tile's buffer, releases each ring stage with tcgen05.commit
//             and commits the buffer after the tile's last K slice;
//   warps 2-5 wait for a buffer's commit, read their 32-lane quarter with
//             tcgen05.ld, release the buffer and run the epilogue: fp32 store,
//             residual add, SwiGLU (gate and up rows paired in one tile),
//             per-head RMSNorm + RoPE + store (dense or into a K/V cache), or a
//             per-row top-2 whose last column tile merges the vocabulary.
// Every wait is bounded; on timeout the CTA flags the status word, drains,
// frees its TMEM and returns.
#include <string.h>

#include "common.cuh"
#include "ptx.cuh"
#include "tc05.cuh"

namespace dflash {

using namespace ptx;

// Tile order.  With few row tiles (a block of drafted rows: 4 at batch 32 x
// B 16) consecutive CTAs take the row tiles of one weight column tile, so
// each weight tile is read from HBM once (column-first order re-read the
// 1.2 GB LM head from HBM once per row tile: 817 -> 560 us at 480 rows);
// with many (a long
// prefix) consecutive CTAs share a row tile of activations instead, which
// measured faster there.  0 keeps column-first order everywhere.
#ifndef DFLASH_TC_MFAST
#define DFLASH_TC_MFAST 1
#endif

constexpr int TC_BM = 128, TC_BK = 64;
constexpr int TC_THREADS = 192;
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;   // 16 KB

// Shared-memory layout of the ring for a BN-column tile.  PAIR: a cluster of
// two CTAs computes a 256-row tile with one tcgen05.mma.cta_group::2 stream
// (issued by the even CTA): each CTA loads its own 128 activation rows and
// half of the tile's weight rows, and holds its 128 rows of the accumulator.
template <int BN, bool PAIR = false>
struct TcCfg {
  static_assert(BN == 128 || BN == 256, "tile width");
  static_assert(!PAIR || BN == 256, "CTA pairs take 256-column tiles");
  static constexpr int BM = PAIR ? 2 * TC_BM : TC_BM;          // rows of a tile
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;           // weight rows a CTA loads per stage
  static constexpr int B_BYTES = B_ROWS * TC_BK * 2;
  static constexpr int STAGE_TX = TC_A_BYTES + B_BYTES;       // bytes a CTA loads per stage
  static constexpr int STAGES = 196608 / STAGE_TX;            // 4 (256), 6 (128 or a pair)
  static constexpr int OFF_B = STAGES * TC_A_BYTES;
  // every TMA load writes exactly one stage: the A box is 128 rows x 64 k,
  // the B box(es) B_ROWS rows (or B_ROWS/2 gate rows + B_ROWS/2 up rows) x
  // 64 k, and each launch pairs the tile with weight maps of that box height
  static constexpr int OFF_BAR = OFF_B + STAGES * B_BYTES;
  static constexpr int SMEM = OFF_BAR + 8 * (2 * STAGES + 4) + 64 + 1024;
  static constexpr uint32_t TMEM_COLS = 2 * BN;   // two accumulators
};
static_assert(TcCfg<256>::SMEM <= 232448 && TcCfg<128>::SMEM <= 232448 &&
                  TcCfg<256, true>::SMEM <= 232448, "shared memory per CTA");

struct TcParams {
  CUtensorMap amap[WS_MAXSRC];
  CUtensorMap bmap[WS_MAXMAP];
  WSeg seg[WS_MAXMAP];
  int nseg, M, K, kc_per_src, n_mtiles, n_ntiles, m_fast;
  RowMap rm;
  const int32_t* len;
  const float2* rope_tab;
  int max_pos;
  float eps;
  int* status;
  float4* amx;          // SK_ARGMAX: top-2 record per (column tile, row)
  int* counters;        // SK_ARGMAX: column tiles finished per row tile
  int32_t* ids;
  float* gap;
  int rps_out;
  const int32_t* anchor;
};
static_assert(sizeof(TcParams) <= 4096, "kernel parameters must fit the 4 KB limit");

__device__ __forceinline__ int tc_seg_of(const TcParams& p, int t) {
  int s = 0;
  while (s + 1 < p.nseg && t >= p.seg[s + 1].t0) ++s;
  return s;
}

// Epilogue of one output tile for the row this thread owns; trow addresses
// the row's TMEM lane in the tile's accumulator.
template <int BN>
__device__ __forceinline__ void tc_tile_epilogue(const TcParams& p, const WSeg& g, int lt, int nt,
                                                 int row, uint32_t trow) {
  constexpr int TC_BN = BN;
  if (g.kind == SK_F32) {
    float* dst = (float*)g.dst;
    for (int c = 0; c < TC_BN / 32; ++c) {
      float v[32];
      tc_ld32(trow + c * 32, v);
      const int n = lt * TC_BN + c * 32;
      if (row < p.M && n < g.n_valid) {
        float4* o = (float4*)(dst + (int64_t)row * g.ld + n);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
    }
  } else if (g.kind == SK_RESID) {
    float* dst = (float*)g.dst;
    for (int c = 0; c < TC_BN / 32; ++c) {
      float v[32];
      tc_ld32(trow + c * 32, v);
      const int n = lt * TC_BN + c * 32;
      if (row < p.M && n < g.n_valid) {
        float4* o = (float4*)(dst + (int64_t)row * g.ld + n);
        float4 old[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) old[i] = o[i];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          o[i] = make_float4(old[i].x + v[4 * i], old[i].y + v[4 * i + 1], old[i].z + v[4 * i + 2],
                             old[i].w + v[4 * i + 3]);
      }
    }
  } else if (g.kind == SK_SWIGLU) {
    bf16* dst = (bf16*)g.dst;
    for (int c = 0; c < TC_BN / 64; ++c) {
      float gv[32], uv[32];
      tc_ld32(trow + c * 32, gv);
      tc_ld32(trow + TC_BN / 2 + c * 32, uv);
      const int f = lt * (TC_BN / 2) + c * 32;
      if (row < p.M && f < g.n_valid) {
        uint4* o = (uint4*)(dst + (int64_t)row * g.ld + f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float a[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float x = gv[8 * i + k];
            a[k] = x / (1.0f + expf(-x)) * uv[8 * i + k];
          }
          __nv_bfloat162 t0 = __floats2bfloat162_rn(a[0], a[1]);
          __nv_bfloat162 t1 = __floats2bfloat162_rn(a[2], a[3]);
          __nv_bfloat162 t2 = __floats2bfloat162_rn(a[4], a[5]);
          __nv_bfloat162 t3 = __floats2bfloat162_rn(a[6], a[7]);
          uint4 w;
          w.x = *reinterpret_cast<uint32_t*>(&t0);
          w.y = *reinterpret_cast<uint32_t*>(&t1);
          w.z = *reinterpret_cast<uint32_t*>(&t2);
          w.w = *reinterpret_cast<uint32_t*>(&t3);
          o[i] = w;
        }
      }
    }
  } else if (g.kind == SK_ARGMAX) {
    // top-2 of this row over the tile's columns (lowest index on ties)
    float t1 = -INFINITY, t2 = -INFINITY;
    int i1 = 0x7fffffff;
    for (int c = 0; c < TC_BN / 32; ++c) {
      float v[32];
      tc_ld32(trow + c * 32, v);
      const int n0 = lt * TC_BN + c * 32;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        if (n0 + k >= g.n_valid) break;
        const float x = v[k];
        if (x > t1) {
          t2 = t1;
          t1 = x;
          i1 = n0 + k;
        } else if (x > t2) {
          t2 = x;
        }
      }
    }
    if (row < p.M) p.amx[(int64_t)nt * p.M + row] = make_float4(t1, __int_as_float(i1), t2, 0.f);
  } else if (g.kind == SK_HEAD && g.d == 128) {
    int b = -1, i = 0;
    const bool mapped = row < p.M && p.rm.map(row, b, i);
    const int pos = mapped ? p.len[b] + i : -1;
    for (int hh = 0; hh < TC_BN / 128; ++hh) {
      float x[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc_ld32(trow + hh * 128 + c * 32, x + 32 * c);
      if (!mapped) continue;
      const int head = lt * (TC_BN / 128) + hh;
      if (g.gain != nullptr) {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 128; ++e) ss += x[e] * x[e];
        const float rinv = 1.0f / sqrtf(ss / 128.0f + p.eps);
#pragma unroll
        for (int e = 0; e < 128; ++e) x[e] = x[e] * rinv * g.gain[e];
      }
      if (g.rope) {
        if (pos < 0 || pos >= p.max_pos) {
          atomicOr(p.status, ST_BOUNDS);
          continue;
        }
        const float2* cs = p.rope_tab + (int64_t)pos * 64;
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const float2 t = cs[e];
          const float y1 = x[e] * t.x - x[e + 64] * t.y;
          const float y2 = x[e + 64] * t.x + x[e] * t.y;
          x[e] = y1;
          x[e + 64] = y2;
        }
      }
      bf16* o;
      if (g.cache_cap > 0) {
        if (b >= g.cache_batch || pos < 0 || pos >= g.cache_cap) {
          atomicOr(p.status, ST_CAPACITY);
          continue;
        }
        o = (bf16*)g.dst + (((int64_t)b * g.cache_heads + head) * g.cache_cap + pos) * 128;
      } else {
        o = (bf16*)g.dst + (int64_t)row * g.ld + (int64_t)head * 128;
      }
#pragma unroll
      for (int e = 0; e < 128; e += 8) {
        uint4 w;
        __nv_bfloat162 t0 = __floats2bfloat162_rn(x[e], x[e + 1]);
        __nv_bfloat162 t1 = __floats2bfloat162_rn(x[e + 2], x[e + 3]);
        __nv_bfloat162 t2 = __floats2bfloat162_rn(x[e + 4], x[e + 5]);
        __nv_bfloat162 t3 = __floats2bfloat162_rn(x[e + 6], x[e + 7]);
        w.x = *reinterpret_cast<uint32_t*>(&t0);
        w.y = *reinterpret_cast<uint32_t*>(&t1);
        w.z = *reinterpret_cast<uint32_t*>(&t2);
        w.w = *reinterpret_cast<uint32_t*>(&t3);
        *reinterpret_cast<uint4*>(o + e) = w;
      }
    }
  }
}

// Top-2 of one row over every column tile's record, in column-tile order
// (lowest index on ties), written as the row's draft id and top-2 gap.
__device__ __forceinline__ void tc_merge_row(const TcParams& p, int row) {
  float t1 = -INFINITY, t2 = -INFINITY;
  int i1 = 0x7fffffff;
  for (int n0 = 0; n0 < p.n_ntiles; n0 += 8) {
    float4 rec[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      rec[k] = (n0 + k < p.n_ntiles) ? __ldcg(&p.amx[(int64_t)(n0 + k) * p.M + row])
                                     : make_float4(-INFINITY, __int_as_float(0x7fffffff), -INFINITY, 0.f);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float a1 = rec[k].x, a2 = rec[k].z;
      const int ai = __float_as_int(rec[k].y);
      const float lo = fminf(t1, a1);
      if (a1 > t1 || (a1 == t1 && ai < i1)) {
        t1 = a1;
        i1 = ai;
      }
      t2 = fmaxf(lo, fmaxf(t2, a2));
    }
  }
  int64_t out = row, gout = row;
  if (p.rps_out > 0) {
    const int per = p.rps_out - 1;
    const int64_t b = row / per, i = row % per + 1;
    out = b * p.rps_out + i;
    gout = b * per + (i - 1);
    if (i == 1) p.ids[b * p.rps_out] = p.anchor[b];
  }
  float g = t1 - t2;
  p.ids[out] = argmax_id(i1, g, p.status);
  if (p.gap) p.gap[gout] = g;
}

// Persistent: CTA c (a pair: cluster c) takes tiles c, c + grid, ... in
// launch order; the ring runs on across its tiles and two TMEM accumulators
// let the epilogue of one tile overlap the MMAs of the next.
template <int BN, bool PAIR>
__global__ void __launch_bounds__(TC_THREADS, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  using C = TcCfg<BN, PAIR>;
  constexpr int TC_STAGES = C::STAGES, TC_B_BYTES = C::B_BYTES;
  constexpr int TC_STAGE_TX = C::STAGE_TX, TC_OFF_B = C::OFF_B, TC_OFF_BAR = C::OFF_BAR;
  constexpr uint32_t TC_TMEM_COLS = C::TMEM_COLS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_u32(smem);
  // ring full / empty per stage; accumulator full (MMA commit) / empty (the
  // four epilogue warps, of both CTAs of a pair) per TMEM buffer
  const uint32_t bar_full = sbase + TC_OFF_BAR, bar_empty = bar_full + 8 * TC_STAGES,
                 bar_tfull = bar_empty + 8 * TC_STAGES, bar_tempty = bar_tfull + 16;
  volatile uint32_t* tmem_slot = (volatile uint32_t*)(smem + TC_OFF_BAR + 8 * (2 * TC_STAGES + 4));
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  volatile int* last_flag = (volatile int*)(tmem_slot + 2);
  volatile int* kcount = (volatile int*)(tmem_slot + 3);   // k-blocks issued, consumed
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // a pair: the even CTA (rank 0) issues the MMAs; the loads of both CTAs
  // complete on its full barriers and both epilogues free its accumulators
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const uint32_t bar_full_l = PAIR ? mapa_shared(bar_full, 0) : bar_full;
  const uint32_t bar_tempty_l = PAIR ? mapa_shared(bar_tempty, 0) : bar_tempty;
  const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int nk = p.K / TC_BK;
  const int tiles = p.n_mtiles * p.n_ntiles;
  const int my_tiles = unit < tiles ? (tiles - 1 - unit) / units + 1 : 0;
  // m_fast: the row tiles that share a weight column tile run side by side,
  // so the column comes from HBM once and from L2 for the others
  auto tile_of = [&](int j, int& mt, int& nt) {
    const int t = unit + j * units;
    mt = p.m_fast ? t % p.n_mtiles : t / p.n_ntiles;
    nt = p.m_fast ? t / p.n_mtiles : t - mt * p.n_ntiles;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < TC_STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, PAIR ? 8 : 4);
    }
    *abort_flag = 0;
    kcount[0] = kcount[1] = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    if (PAIR) {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32((const void*)tmem_slot)),
                   "r"(TC_TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32((const void*)tmem_slot)),
                   "r"(TC_TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();   // both CTAs' barriers and TMEM exist before either signals the other
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ---- producer -------------------------------------------------------------
      // the operand other CTAs read again later stays in L2: the activations
      // when consecutive CTAs share a weight column tile (every column tile
      // re-reads them), the weights otherwise
      const uint64_t pol_w = p.m_fast ? policy_evict_first() : policy_evict_last();
      const uint64_t pol_a = p.m_fast ? policy_evict_last() : policy_evict_first();
      auto load = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                      uint64_t pol) {
        if (PAIR) tma_load_2d_pair(dst, map, bar, c0, c1, pol);
        else tma_load_2d(dst, map, bar, c0, c1, pol);
      };
      pdl_wait();
      int kg = 0;   // k-blocks issued over this CTA's tiles
      for (int j = 0; j < my_tiles && !*abort_flag; ++j) {
        int mt, nt;
        tile_of(j, mt, nt);
        const WSeg& g = p.seg[tc_seg_of(p, nt)];
        const int lt = nt - g.t0;
        const int arow = mt * C::BM + (int)rank * TC_BM;
        for (int kb = 0; kb < nk; ++kb, ++kg) {
          const int s = kg % TC_STAGES, use = kg / TC_STAGES;
          if (use > 0 && !mbar_wait(bar_empty + 8 * s, (use - 1) & 1)) {
            atomicOr(p.status, ST_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          if (*abort_flag) break;
          if (rank == 0) mbar_arrive_expect_tx(bar_full + 8 * s, (PAIR ? 2 : 1) * TC_STAGE_TX);
          const uint32_t fb = bar_full_l + 8 * s;
          const int src = kb / p.kc_per_src, lk = kb - src * p.kc_per_src;
          load(sbase + s * TC_A_BYTES, &p.amap[src], fb, lk * TC_BK, arow, pol_a);
          const uint32_t bdst = sbase + TC_OFF_B + s * TC_B_BYTES;
          if (g.kind == SK_SWIGLU) {
            // gate and up rows of the tile's BN/2 FFN columns: a pair's even
            // CTA loads the gate rows, the odd one the up rows
            if (PAIR) {
              load(bdst, &p.bmap[rank ? g.map2 : g.map], fb, kb * TC_BK, lt * (BN / 2), pol_w);
            } else {
              load(bdst, &p.bmap[g.map], fb, kb * TC_BK, lt * (BN / 2), pol_w);
              load(bdst + TC_B_BYTES / 2, &p.bmap[g.map2], fb, kb * TC_BK, lt * (BN / 2), pol_w);
            }
          } else {
            load(bdst, &p.bmap[g.map], fb, kb * TC_BK, lt * BN + (int)rank * C::B_ROWS, pol_w);
          }
        }
      }
      kcount[0] = kg;
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---- MMA issuer: tile j accumulates into TMEM buffer j & 1 -----------------
      const uint32_t idesc = idesc_bf16_f32(C::BM, BN);
      int kg = 0;   // k-blocks consumed
      for (int j = 0; j < my_tiles; ++j) {
        const int b = j & 1, ub = j >> 1;
        if (*abort_flag) break;
        // the epilogue(s) of tile j - 2 have read this buffer
        if (ub > 0 && !mbar_wait(bar_tempty + 8 * b, (ub - 1) & 1)) {
          atomicOr(p.status, ST_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(b * BN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++kg) {
          const int s = kg % TC_STAGES, use = kg / TC_STAGES;
          if (*abort_flag || !mbar_wait(bar_full + 8 * s, use & 1)) {
            atomicOr(p.status, ST_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sbase + s * TC_A_BYTES, b0 = sbase + TC_OFF_B + s * TC_B_BYTES;
#pragma unroll
          for (int jj = 0; jj < TC_BK / 16; ++jj) {
            const uint32_t accum = (kb > 0 || jj > 0) ? 1u : 0u;
            if (PAIR) tc_mma2(acc, sdesc_sw128(a0 + jj * 32), sdesc_sw128(b0 + jj * 32), idesc, accum);
            else tc_mma(acc, sdesc_sw128(a0 + jj * 32), sdesc_sw128(b0 + jj * 32), idesc, accum);
          }
          if (PAIR) tc_commit2(bar_empty + 8 * s);
          else tc_commit(bar_empty + 8 * s);
        }
        if (!ok) break;
        if (PAIR) tc_commit2(bar_tfull + 8 * b);
        else tc_commit(bar_tfull + 8 * b);
      }
      kcount[1] = kg;
    }
    __syncwarp();
  } else {
    // ---- epilogue: warps 2-5, TMEM lane quarter (warp % 4) -----------------------
    // Every warp walks all of the CTA's tiles (after an abort without waiting),
    // so the four warps always meet at the same named barriers.
    pdl_wait();                                     // cache lengths come from earlier kernels
    const int q = warp & 3;
    const int r = q * 32 + lane;                    // row within this CTA's 128 rows of the tile
    for (int j = 0; j < my_tiles; ++j) {
      const int b = j & 1, ub = j >> 1;
      int mt, nt;
      tile_of(j, mt, nt);
      const WSeg& g = p.seg[tc_seg_of(p, nt)];
      const int lt = nt - g.t0;
      const int rt = mt * (C::BM / TC_BM) + (int)rank;   // this CTA's 128-row tile
      const int row = rt * TC_BM + r;
      const bool ok = !(*abort_flag & 1) && mbar_wait(bar_tfull + 8 * b, ub & 1, 4000000000ull);
      if (!ok && !(*abort_flag & 1)) {
        atomicOr(p.status, ST_TIMEOUT);
        *abort_flag = 1;
      }
      tc_fence_after();
      if (ok) tc_tile_epilogue<BN>(p, g, lt, nt, row, tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR) mbar_arrive_cluster(bar_tempty_l + 8 * b);
        else mbar_arrive(bar_tempty + 8 * b);
      }
      if (g.kind == SK_ARGMAX) {
        // the CTA that finishes the last column tile of this 128-row tile
        // merges the records of its rows over all column tiles
        __threadfence();
        named_bar(1, 128);
        if (warp == 2 && lane == 0) {
          const int old = atomicAdd(&p.counters[rt], 1);
          const int last = (old == p.n_ntiles - 1);
          if (last) p.counters[rt] = 0;
          *last_flag = last;
        }
        named_bar(1, 128);
        if (*last_flag) {
          __threadfence();
          if (row < p.M) tc_merge_row(p, row);
        }
        named_bar(1, 128);   // the flag is read before the next tile rewrites it
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if ((*abort_flag & 1) && threadIdx.x == 0) {
    if (PAIR) {
      // loads of this CTA may still be in flight, counted on the even CTA's
      // barriers: give them time to land (bounded) before shared memory goes
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < 200000ull) __nanosleep(1000);
    } else {
      // let the TMA loads still in flight land and the issued MMAs finish
      // before the shared memory and TMEM are released (each wait bounded)
      const int issued = kcount[0], used = kcount[1];
      for (int i = used; i < issued && i < used + TC_STAGES; ++i)
        mbar_wait(bar_full + 8 * (i % TC_STAGES), (i / TC_STAGES) & 1, 20000000ull);
      if (used > 0)
        mbar_wait(bar_empty + 8 * ((used - 1) % TC_STAGES), ((used - 1) / TC_STAGES) & 1, 20000000ull);
    }
  }
  if (PAIR) {
    // neither CTA leaves while the other may still arrive on its barriers or
    // the even CTA's MMAs may still use the odd CTA's TMEM
    __syncthreads();
    cluster_sync();
  }
  if (warp == 1) {
    tc_fence_after();
    if (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                   "r"(TC_TMEM_COLS)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                   "r"(TC_TMEM_COLS)
                   : "memory");
  }
}

// ---------------------------------------------------------------------------
// The three variants: 256-column tiles, 128-column tiles, 256-row x 256-column
// tiles on CTA pairs.
using TcKernel = void (*)(TcParams);
static TcKernel tc_kernel(int bi) {
  return bi == 2 ? tc_gemm_kernel<256, true> : bi == 1 ? tc_gemm_kernel<128, false>
                                                       : tc_gemm_kernel<256, false>;
}
static int tc_smem(int bi) {
  return bi == 2 ? TcCfg<256, true>::SMEM : bi == 1 ? TcCfg<128>::SMEM : TcCfg<256>::SMEM;
}
static cudaError_t tc_set_smem(int bi) {
  static bool done[3] = {false, false, false};
  if (done[bi]) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(tc_kernel(bi), cudaFuncAttributeMaxDynamicSharedMemorySize, tc_smem(bi));
  done[bi] = e == cudaSuccess;
  return e;
}

// CTA pairs that can be resident at once (0: clusters unavailable).
int tc_pair_units(const dflash_handle* h) {
  static int units = -1;
  if (units >= 0) return units;
  units = 0;
  if (tc_set_smem(2) != cudaSuccess) return units;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * std::max(1, h->num_sms / 2));
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = tc_smem(2);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_kernel(2), &cfg) == cudaSuccess && n > 0)
    units = std::min(n, h->num_sms / 2);
  cudaGetLastError();
  return units;
}

int tc_gemm(dflash_handle* h, cudaStream_t s, int kclass, const WLaunch& L, float4* amx) {
  if ((L.bn != 128 && L.bn != 256) || L.M < 1 || L.K % TC_BK != 0 || L.nseg < 1 ||
      L.nseg > WS_MAXMAP || L.nsrc < 1 || L.nsrc > WS_MAXSRC || (L.K / TC_BK) % L.nsrc != 0)
    return DFLASH_ERR_SHAPE;
  for (int i = 0; i < L.nseg; ++i)
    if (L.seg[i].kind == SK_HEAD && L.seg[i].d != 128) return DFLASH_ERR_SHAPE;
  TcParams prm;
  memset(&prm, 0, sizeof(prm));
  const int kc_per_src = L.K / TC_BK / L.nsrc;
  for (int i = 0; i < L.nsrc; ++i)
    if (!make_tmap_2d(&prm.amap[i], L.a_src[i], (uint64_t)kc_per_src * TC_BK, (uint64_t)L.M,
                      (uint64_t)L.a_ld * 2, TC_BK, TC_BM))
      return DFLASH_ERR_CUDA;
  for (int i = 0; i < L.nmap; ++i) prm.bmap[i] = *L.wmaps[i];
  for (int i = 0; i < L.nseg; ++i) prm.seg[i] = L.seg[i];
  prm.nseg = L.nseg;
  prm.M = L.M;
  prm.K = L.K;
  prm.kc_per_src = kc_per_src;
  // CTA pairs (256-column tiles; the caller's weight maps have boxes of 128
  // rows, half a tile)
  const bool pair = L.pair;
  if (pair && (L.bn != 256 || tc_pair_units(h) <= 0)) return DFLASH_ERR_SHAPE;
  const int bm = pair ? 2 * TC_BM : TC_BM;
  prm.n_ntiles = L.seg[L.nseg - 1].t1;
  prm.n_mtiles = (L.M + bm - 1) / bm;
  prm.m_fast = DFLASH_TC_MFAST && prm.n_mtiles * 8 <= (pair ? tc_pair_units(h) : h->num_sms);
  prm.rm = L.rm;
  prm.len = L.len;
  prm.rope_tab = h->d_rope;
  prm.max_pos = h->cfg.max_pos;
  prm.eps = h->cfg.rms_eps;
  prm.status = h->d_status;
  prm.amx = amx;
  prm.counters = h->d_counters;
  prm.ids = L.ids;
  prm.gap = L.gap;
  prm.rps_out = L.rps_out;
  prm.anchor = L.anchor;
  const int64_t tiles = (int64_t)prm.n_mtiles * prm.n_ntiles;
  if (L.seg[0].kind == SK_ARGMAX && (prm.n_mtiles * (bm / TC_BM) > kMaxTiles || !amx))
    return DFLASH_ERR_SHAPE;
  if (tiles > 0x7fffffff) return DFLASH_ERR_SHAPE;
  const int bi = pair ? 2 : L.bn == 128 ? 1 : 0;
  if (tc_set_smem(bi) != cudaSuccess) return DFLASH_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  // persistent: one CTA per SM (its shared memory admits no second), each
  // CTA (or pair of CTAs) walking every grid-th tile
  const int64_t units = pair ? std::min<int64_t>(tiles, tc_pair_units(h))
                             : std::min<int64_t>(tiles, h->num_sms);
  cfg.gridDim = dim3((unsigned)(pair ? 2 * units : units));
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = tc_smem(bi);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pair ? 2 : 1;
  auto kern = tc_kernel(bi);
  Timer t;
  launch_begin(h, kclass, s, &t);
  cudaLaunchKernelEx(&cfg, kern, prm);
  return launch_end(h, s, &t);
}

}  // namespace dflash
