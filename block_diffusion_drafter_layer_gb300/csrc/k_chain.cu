// Persistent draft-block kernel for short blocks (at most 16 rows in all).
//
// A draft block of one sequence (or a few short ones) multiplies a handful of
// rows by every draft weight, so its time is the time to read those weights
// from HBM.  Issued as one launch per projection, each launch loses several
// microseconds to start-up, ramp and the split-K fix-up tail.  This kernel
// runs the whole block (txtmix §6: embed the block [anchor, mask, ...], the
// draft layers over [context ; block], the shared LM head) in one cooperative
// launch of two CTAs per SM, as a fixed sequence of phases separated by
// grid-wide barriers:
//
//   embed | per layer: q/k/v  attention  combine  o_proj  gate/up  down | LM head
//
// (each projection followed by a reduce phase, below)
//
// * Projections stream their weight tiles through a TMA / mbarrier ring in
//   (128-row tile, 64-column chunk) units spread evenly over the CTAs (split
//   K).  A CTA finishes the tiles it owns whole; for the others it leaves a
//   partial sum, and the following reduce phase gives each (tile, row) to one
//   warp, which adds the partials in k order and runs the epilogue.  The
//   producer lane keeps loading the NEXT projection's weights while the grid
//   waits at a barrier (weights do not depend on activations); only the
//   activation loads wait for the barrier.
// * The RMSNorms in front of q/k/v, gate/up and the LM head are folded into
//   those projections' operand loads.  The residual epilogues (and the
//   embedding) write the residual x, x * g in fp32 for the next norm's gain
//   g, and one sum of squares of x per (128-column tile, row).  The next
//   projection takes 1 / rms of each row from those sums at its start
//   (while its first fp32 (x * g) chunks are in flight) and its MMA warps
//   round each chunk to bf16(x * g / rms) — the normalised row at the same
//   storage point as a separate RMSNorm — before they multiply it.
// * Attention cuts the keys of each (sequence, kv head) into equal runs of
//   32-key sub-chunks, one run per work item, items dealt round-robin to the
//   CTAs; each item keeps (max, sum, unnormalised output) per query row, and
//   the combine phase merges the runs of a row in run order.
//
// Every wait is bounded; a CTA that gives up sets ST_TIMEOUT, which every
// other CTA polls while it waits, so the grid drains within one wait limit.
#include <string.h>

#include "common.cuh"
#include "ptx.cuh"

namespace dflash {

using namespace ptx;

#ifndef DFLASH_CH_STAGES
#define DFLASH_CH_STAGES 5
#endif
// attention probabilities enter P V as a bf16 (hi, lo) pair (1) or as bf16 (0)
#ifndef DFLASH_CH_PLO
#define DFLASH_CH_PLO 1
#endif
// pause of the producer lane between polls when nothing can be issued (ns)
#ifndef DFLASH_CH_IDLE_NS
#define DFLASH_CH_IDLE_NS 64
#endif

// warp 0: TMA producer; warps 1-4: consumers; warp 5 only waits at the
// kernel's final barrier.  The sixth warp measured 6 us faster per
// Qwen3-8B-shaped round than five (same code otherwise, alternating builds),
// with the register budget of 192 threads (below) also keeping every value
// in registers; the likely cause is where the two CTAs' warps, the producers
// among them, land on the SM's four sub-partitions.
constexpr int CH_THREADS = 192;
constexpr int CH_CT = 128;                 // consumer threads
constexpr int CH_STAGES = DFLASH_CH_STAGES;
constexpr int CH_W = 128 * 64 * 2;         // weight chunk: 128 rows x 64 k, bf16
constexpr int CH_A = 16 * 64 * 2;          // activation chunk: 16 rows x 64 k, bf16
constexpr int CH_AF = 16 * 64 * 4;         // fp32 (x * g) chunk of a normalised operand
constexpr int CH_AS = CH_AF;               // ring bytes per activation stage
constexpr int CH_DH = 128;                 // head dim of the attention phases
constexpr int CH_AK = 32;                  // keys per attention sub-chunk
constexpr int CH_DP = CH_DH + 4;           // attention partial row: max, sum, 2 pad, output
constexpr int CH_EPAD = 132;               // fp32 tile row pitch in shared memory
constexpr int CH_ROWS = 16;                // rows of the block (all sequences)
constexpr int CH_MAXB = 16;                // sequences
// floats between consecutive sums of squares: each (tile, row) value is
// written by a different warp, so each gets a 32-byte sector of its own
#ifndef DFLASH_CH_SSQ_STRIDE
#define DFLASH_CH_SSQ_STRIDE 8
#endif
constexpr int CH_SSQ = DFLASH_CH_SSQ_STRIDE;

// shared memory layout (offsets from a 1024-aligned base).  The attention
// phases use the ring's memory: the producer loads no weight unit of a phase
// after attention(l) until this CTA has finished attention(l), and every
// earlier ring entry has been consumed before attention(l) starts.
constexpr int CH_OFF_A = CH_STAGES * CH_W;
constexpr int CH_RING_BYTES = CH_OFF_A + CH_STAGES * CH_AS;
constexpr int CH_OFF_ATT = 0;
constexpr int CH_ATT_Q = 64 * CH_DH * 2;              // 64 query rows
constexpr int CH_ATT_KV = CH_AK * CH_DH * 2;          // one K (or V) sub-chunk
constexpr int CH_ATT_BYTES = CH_ATT_Q + 4 * CH_ATT_KV; // Q + 2 stages x (K, V)
constexpr int CH_OFF_E = CH_RING_BYTES;               // fp32 output tile [16][CH_EPAD]
constexpr int CH_OFF_BAR = CH_OFF_E + CH_ROWS * CH_EPAD * 4;   // full, empty per stage
constexpr int CH_OFF_MISC = CH_OFF_BAR + 2 * CH_STAGES * 8;
constexpr int CH_MISC_BYTES = 2048;
constexpr int CH_SMEM = CH_OFF_MISC + CH_MISC_BYTES + 1024;
static_assert(CH_ATT_BYTES <= CH_RING_BYTES, "the attention buffers alias the ring");
static_assert(2 * CH_A <= CH_ROWS * CH_EPAD * 4, "the rounded operand buffers alias E");
static_assert(CH_SMEM <= 233472 / 2 - 1024, "two CTAs per SM");

enum ChainPhase : int {
  PH_EMBED, PH_QKV, PH_ATT, PH_CMB, PH_O, PH_GU, PH_DN, PH_LM, PH_RED, PH_LMFIN,
  PH_FUSE, PH_FNORM, PH_INJ   // the round's context projection, its norm, the K/V injection
};
// phases of one layer; every projection is followed by its reduce phase
constexpr int kLayerPhases = 10;
__device__ __constant__ const int kLayerSeq[kLayerPhases] = {PH_QKV, PH_RED, PH_ATT, PH_CMB, PH_O,
                                                             PH_RED, PH_GU,  PH_RED, PH_DN,  PH_RED};
// phases a round runs before the draft block: fuse the pending target
// features, normalise them, inject their K/V into every layer's cache
constexpr int kRoundPhases = 5;
__device__ __constant__ const int kRoundSeq[kRoundPhases] = {PH_FUSE, PH_RED, PH_FNORM, PH_INJ, PH_RED};

struct ChainLayer {
  const float* g_in;
  const float* g_post;
  const float* q_norm;
  const float* k_norm;
};

struct ChainParams {
  CUtensorMap map_hid[DFLASH_MAX_PICK];   // round: the pending target features [n_in, D], box 64 x 16
  CUtensorMap map_ht;         // round: the fused context feature H_t [n_in, D], box 64 x 16
  CUtensorMap map_xg;         // fp32 x * g [R, D], box 64 x 16, unswizzled
  CUtensorMap map_o;          // bf16 attention output [R, H*d], box 64 x 16
  CUtensorMap map_a;          // bf16 SwiGLU output [R, F], box 64 x 16
  const CUtensorMap* wmaps;   // [n_layers * 7 + 2]: q k v o gate up down per layer, LM head, W_c
  const bf16* kc[DFLASH_MAX_LAYERS];
  const bf16* vc[DFLASH_MAX_LAYERS];
  ChainLayer lay[DFLASH_MAX_LAYERS];
  const bf16* embed;
  const float* g_f;
  const float* g_c;           // round: the fused context's RMSNorm gain
  bf16* ht;                   // round: H_t out [n_in, D]
  const int32_t* row0;        // round: first pending row of each sequence
  const int32_t* nrow;        // round: pending rows of each sequence (appended to its cache)
  const int32_t* anchor;
  int32_t* len;               // cache lengths (a round advances them)
  int32_t* ids;
  float* gap;
  float* x;
  float* xg;
  bf16* q;
  bf16* kb;
  bf16* vb;
  bf16* o;
  bf16* a;
  float* ssq;                 // [D / 128][16] rows, CH_SSQ floats apart
  float* partial;             // split-K fix-up: [2 * grid][16 * 128]
  float* apart;               // attention items: [n_items_max][64][CH_DP]
  float4* amx;                // LM-head top-2 records: [vocab tiles][R]
  int* counters;              // grid barrier at kMaxTiles + 1
  int* status;
  unsigned long long* trace;  // optional: kChainTraceCols arrays of [kChainMaxPhases] (ns)
  const float2* rope;
  int max_pos;
  int R, batch, B, D, Hd, Gd, F, V, G, rep, nL, cap, mask_id, qk_norm;
  int pre, n_in, n_pick, kv_batch;   // round phases (0 or kRoundPhases), pending rows, sources, cache batch
  int grid, n_phases, n_items_max;
  float eps, embed_scale, scale_log2;
  int causal_layers, window_layers, window;   // draft layer types (bit l: layer l)
};
static_assert(sizeof(ChainParams) <= 4096, "kernel parameters must fit the 4 KB limit");

// misc words in shared memory
// MS_ABORT may be set by any thread at any time; MS_GO and MS_LAST are
// written by consumer thread 0 only between two consumer barriers, so every
// consumer warp reads the same value and takes the same barriers.
// MS_ATT_DONE: layers whose attention phase this CTA has finished (written by
// consumer thread 0, read by the producer).
enum : int { MS_ABORT = 0, MS_LAST = 1, MS_ISSUED = 2, MS_CONSUMED = 3, MS_GO = 4, MS_ATT_DONE = 5 };
// [0, 16) ints: flags; [16, 48): rowpos (sequence, position) per row;
// [48, 64): 1 / rms per row; [64, 192): attention item tables; [192, 384):
// LM-head top-2 records, [4 warps][16 rows][3]; [384, 416): injpos
// (sequence, cache position) per pending row of a round

// Phase p: the round's phases (p < P.pre), then embed; kLayerPhases per
// layer; the LM head, its reduce (which also publishes each CTA's top-2
// records) and the final merge.
template <bool RD>
__device__ __forceinline__ int phase_kind(const ChainParams& P, int p, int& l) {
  if (RD && p < P.pre) {
    l = 0;
    return kRoundSeq[p];
  }
  if (RD) p -= P.pre;
  if (p == 0) {
    l = 0;
    return PH_EMBED;
  }
  const int q = p - 1;
  l = q / kLayerPhases;
  if (l >= P.nL) {
    l = P.nL;
    const int k = q - P.nL * kLayerPhases;
    return k == 0 ? PH_LM : k == 1 ? PH_RED : PH_LMFIN;
  }
  return kLayerSeq[q % kLayerPhases];
}

// nin: the phase's input RMSNorm is folded in (its operand arrives as fp32
// x * g and is rounded to bf16(x * g / rms(x)) in shared memory)
struct Geo {
  int n_tiles, kc, nin;
};
__device__ __forceinline__ Geo gemm_geo(const ChainParams& P, int kind) {
  switch (kind) {
    case PH_QKV: return {(P.Hd + 2 * P.Gd) / 128, P.D / 64, 1};
    case PH_O: return {P.D / 128, P.Hd / 64, 0};
    case PH_GU: return {P.F / 64, P.D / 64, 1};
    case PH_DN: return {P.D / 128, P.F / 64, 0};
    case PH_FUSE: return {P.D / 128, P.n_pick * (P.D / 64), 0};
    case PH_INJ: return {P.nL * 2 * (P.Gd / 128), P.D / 64, 0};   // per layer: k tiles, v tiles
    default: return {(P.V + 127) / 128, P.D / 64, 1};   // PH_LM
  }
}
template <bool RD>
__device__ __forceinline__ bool is_gemm(int kind) {
  return kind == PH_QKV || kind == PH_O || kind == PH_GU || kind == PH_DN || kind == PH_LM ||
         (RD && (kind == PH_FUSE || kind == PH_INJ));
}
// rows of a phase's activations: the round's pending rows or the block rows
template <bool RD>
__device__ __forceinline__ int rows_of(const ChainParams& P, int kind) {
  return RD && (kind == PH_FUSE || kind == PH_INJ) ? P.n_in : P.R;
}

__device__ __forceinline__ int first_unit_of(int64_t c, int64_t U, int64_t G) {
  return (int)(c * U / G);
}
__device__ __forceinline__ int owner_of(int64_t u, int64_t U, int64_t G) {
  return (int)(((u + 1) * G + U - 1) / U) - 1;
}

// Trace helper: latest time over the grid for column `col` of phase `p`.
__device__ __forceinline__ void trace_max(const ChainParams& P, int col, int p) {
  if (P.trace != nullptr) atomicMax(P.trace + col * kChainMaxPhases + p, (unsigned long long)globaltimer());
}

#ifndef DFLASH_CH_EVLOG
#define DFLASH_CH_EVLOG 0
#endif
// Event log of sampled CTAs (every grid/4-th), compiled in on request only.
// Times are the SM's cycle counter (exact within one CTA; %globaltimer ticks
// too coarsely for sub-microsecond steps), so compare events of one CTA only.
__device__ __forceinline__ void ev(const ChainParams& P, int p, int slot) {
  if (DFLASH_CH_EVLOG && P.trace != nullptr) {
    const int q = P.grid / kEvCtas;
    if (q > 0 && blockIdx.x % q == 0 && blockIdx.x / q < kEvCtas && slot < kEvSlots)
      P.trace[(size_t)kChainTraceCols * kChainMaxPhases +
              ((size_t)(blockIdx.x / q) * kChainMaxPhases + p) * kEvSlots + slot] = clock64();
  }
}

// This CTA's units [u0, u1) of a projection phase: an even share of all
// (tile, k-chunk) units (split K).  (Dealing the LM head's 1187 tiles out
// whole instead, to leave nothing to reduce, made that phase 12% slower.)
__device__ __forceinline__ void unit_range(const ChainParams& P, int kind, int cta, int& u0, int& u1) {
  const Geo g = gemm_geo(P, kind);
  const int64_t U = (int64_t)g.n_tiles * g.kc;
  u0 = first_unit_of(cta, U, P.grid);
  u1 = first_unit_of(cta + 1, U, P.grid);
}

// ---- grid barrier ----------------------------------------------------------
// Phase p may start once every CTA has arrived p times.  Gives up (and flags
// ST_TIMEOUT) after the wall-clock limit or as soon as another CTA has.
__device__ bool grid_wait(const ChainParams& P, int target) {
  return bounded_wait_geq(P.counters + kMaxTiles + 1, target, P.status, ST_TIMEOUT,
                          2000000000ull, 0);
}

// ---- producer ----------------------------------------------------------------
// One lane walks this CTA's projection units of every phase twice: a weight
// cursor that fills ring slots as soon as they are free, and an activation
// cursor that follows it once the unit's phase has passed its barrier.
struct Cursor {
  int p, kind, l, u, u1, kc;
  int i;        // ring index
  int t, kk;    // tile and k-chunk of unit u
  const CUtensorMap* wm0;   // weight box(es) of tile t (gate / up: two)
  const CUtensorMap* wm1;
  int wrow;     // row coordinate of tile t in its weight
  // set when the cursor enters a phase: the activation map of k-chunk kk is
  // amap[asrc] at column alk * 64 (asrc steps every aper k-chunks: the
  // fusion's sources), and the attention phases the unit's weights wait for
  const CUtensorMap* amap;
  int aper, asrc, alk, att_need;
  int abytes;   // activation bytes of a unit: CH_AF (fp32 x * g) or CH_A (bf16)
};

// Weight map(s) and row of the cursor's tile.
template <bool RD>
__device__ __forceinline__ void cursor_tile(const ChainParams& P, Cursor& c) {
  c.wm1 = nullptr;
  if (c.kind == PH_LM) {
    c.wm0 = P.wmaps + P.nL * 7;
    c.wrow = c.t * 128;
    return;
  }
  if (RD && c.kind == PH_FUSE) {
    c.wm0 = P.wmaps + P.nL * 7 + 1;
    c.wrow = c.t * 128;
    return;
  }
  if (RD && c.kind == PH_INJ) {   // layer t / 2tk; its k tiles, then its v tiles
    const int tk = P.Gd / 128, li = c.t / (2 * tk), w = (c.t - li * 2 * tk) / tk;
    c.wm0 = P.wmaps + li * 7 + 1 + w;
    c.wrow = (c.t - li * 2 * tk - w * tk) * 128;
    return;
  }
  const CUtensorMap* L = P.wmaps + c.l * 7;
  switch (c.kind) {
    case PH_QKV: {
      const int tq = P.Hd / 128, tk = P.Gd / 128;
      const int w = c.t < tq ? 0 : c.t < tq + tk ? 1 : 2;
      c.wm0 = L + w;
      c.wrow = (c.t - (w == 0 ? 0 : w == 1 ? tq : tq + tk)) * 128;
      break;
    }
    case PH_O: c.wm0 = L + 3; c.wrow = c.t * 128; break;
    case PH_GU:
      c.wm0 = L + 4;
      c.wm1 = L + 5;
      c.wrow = c.t * 64;
      break;
    default: c.wm0 = L + 6; c.wrow = c.t * 128; break;   // PH_DN
  }
}

template <bool RD>
__device__ __forceinline__ bool cursor_phase(const ChainParams& P, Cursor& c, int p) {
  for (; p < P.n_phases; ++p) {
    int l;
    const int kind = phase_kind<RD>(P, p, l);
    if (!is_gemm<RD>(kind)) continue;
    const Geo g = gemm_geo(P, kind);
    int u0, u1;
    unit_range(P, kind, blockIdx.x, u0, u1);
    if (u1 <= u0) continue;
    c.p = p;
    c.kind = kind;
    c.l = l;
    c.u = u0;
    c.u1 = u1;
    c.kc = g.kc;
    c.t = u0 / g.kc;
    c.kk = u0 - c.t * g.kc;
    cursor_tile<RD>(P, c);
    if (RD && kind == PH_FUSE) {
      c.amap = P.map_hid;
      c.aper = P.D / 64;
    } else {
      c.amap = kind == PH_O ? &P.map_o : kind == PH_DN ? &P.map_a
               : RD && kind == PH_INJ ? &P.map_ht : &P.map_xg;
      c.aper = g.kc;
    }
    c.asrc = c.kk / c.aper;
    c.alk = c.kk - c.asrc * c.aper;
    c.abytes = g.nin ? CH_AF : CH_A;
    // ring memory doubles as the attention buffers: a weight unit may be
    // loaded only once this CTA has finished every attention phase before
    // the unit's phase (q/k/v(l) follows attention(l-1); o_proj(l) onward
    // follows attention(l); the LM head follows them all)
    c.att_need = kind == PH_QKV || (RD && (kind == PH_FUSE || kind == PH_INJ)) ? l
                 : kind == PH_LM ? P.nL : l + 1;
    return true;
  }
  c.p = P.n_phases;
  return false;
}
template <bool RD>
__device__ __forceinline__ bool cursor_next(const ChainParams& P, Cursor& c) {
  ++c.i;
  if (++c.u >= c.u1) return cursor_phase<RD>(P, c, c.p + 1);
  if (++c.alk == c.aper) {
    c.alk = 0;
    ++c.asrc;
  }
  if (++c.kk == c.kc) {
    c.kk = 0;
    c.asrc = c.alk = 0;
    ++c.t;
    cursor_tile<RD>(P, c);
  }
  return true;
}

__device__ __forceinline__ void issue_w(const ChainParams& P, const Cursor& c, uint32_t dst,
                                        uint32_t bar, uint64_t pol) {
  tma_load_2d(dst, c.wm0, bar, c.kk * 64, c.wrow, pol);
  if (c.wm1 != nullptr) tma_load_2d(dst + CH_W / 2, c.wm1, bar, c.kk * 64, c.wrow, pol);
}

__device__ __forceinline__ void issue_a(const ChainParams& P, const Cursor& c, uint32_t dst,
                                        uint32_t bar, uint64_t pol) {
  tma_load_2d(dst, c.amap + c.asrc, bar, c.alk * 64, 0, pol);
}

template <bool RD>
__device__ void producer(const ChainParams& P, uint32_t sbase, uint32_t bar_full,
                         uint32_t bar_empty, volatile int* misc) {
  const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
  Cursor w{}, a{};
  w.i = a.i = 0;
  bool w_more = cursor_phase<RD>(P, w, 0);
  a = w;
  bool a_more = w_more;
  int ready = 0;                 // phases known to have passed their barrier
  uint64_t t_idle = 0;
  uint32_t idle = 0;
  bool abort = false;
  while (a_more) {
    bool prog = false;
    const bool w_held = w_more && misc[MS_ATT_DONE] < w.att_need;
    if (w_more && !abort && !w_held) {
      const int s = w.i % CH_STAGES, use = w.i / CH_STAGES;
      // with no activation load owed, block in the barrier wait instead of spinning
      if (use == 0 || (a.i == w.i ? mbar_try_wait(bar_empty + 8 * s, (use - 1) & 1)
                                  : mbar_test_wait(bar_empty + 8 * s, (use - 1) & 1))) {
        mbar_arrive_expect_tx(bar_full + 8 * s, CH_W + w.abytes);
        issue_w(P, w, sbase + s * CH_W, bar_full + 8 * s, pol_w);
        if (DFLASH_CH_EVLOG) {
          int e0, e1;
          unit_range(P, w.kind, blockIdx.x, e0, e1);
          const int k = w.u - e0;
          if (k < kEvUnits) ev(P, w.p, 2 + 2 * kEvUnits + k);
        }
        w_more = cursor_next<RD>(P, w);
        prog = true;
      }
    }
    if (a.i < w.i) {
      bool ok = abort || a.p <= ready;
      if (!ok && ld_acquire_gpu(P.counters + kMaxTiles + 1) >= a.p * P.grid) {
        // the phase's inputs are visible to this thread; order them before
        // its TMA (async-proxy) reads
        fence_proxy_async_global();
        ready = a.p;
        ok = true;
      }
      if (ok) {
        const int s = a.i % CH_STAGES;
        issue_a(P, a, sbase + CH_OFF_A + s * CH_AS, bar_full + 8 * s, pol_a);
        if (DFLASH_CH_EVLOG) {
          int e0, e1;
          unit_range(P, a.kind, blockIdx.x, e0, e1);
          const int k = a.u - e0;
          if (k < kEvUnits) ev(P, a.p, 2 + 3 * kEvUnits + k);
        }
        a_more = cursor_next<RD>(P, a);
        prog = true;
      }
    } else if (!w_more) {
      break;   // every issued unit has its activation load
    }
    if (prog) {
      t_idle = 0;
      idle = 0;
      continue;
    }
    if (abort) break;   // nothing left that can complete
    // idle: give the issue slots to the consumer warps sharing this SM sub-partition
    __nanosleep(w_held && a.i == w.i ? 256 : DFLASH_CH_IDLE_NS);
    // the abort flags and the clock are checked every 64th idle turn only:
    // a global load here would hold the lane for a microsecond each turn
    if ((++idle & 63) != 0) continue;
    if (misc[MS_ABORT] || (*(volatile int*)P.status & ST_TIMEOUT)) {
      abort = true;     // stop loading weights; finish the activation loads already owed
      continue;
    }
    const uint64_t now = globaltimer();
    if (t_idle == 0) t_idle = now;
    else if (now - t_idle > 2000000000ull) {
      atomicOr(P.status, ST_TIMEOUT);
      misc[MS_ABORT] = 1;
      abort = true;
    }
  }
  misc[MS_ISSUED] = w.i;
}

// ---- consumers: projection ------------------------------------------------------
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
__device__ __forceinline__ float4 shfl_xor4(float4 v, int m) {
  return make_float4(__shfl_xor_sync(0xffffffffu, v.x, m), __shfl_xor_sync(0xffffffffu, v.y, m),
                     __shfl_xor_sync(0xffffffffu, v.z, m), __shfl_xor_sync(0xffffffffu, v.w, m));
}

// Row epilogues.  One warp finishes one row r of one output tile t; lane k
// holds the tile's columns 4k .. 4k+3.  Global inputs of the epilogue are
// fetched first (row_in) so their latency overlaps the partial-tile loads.
struct RowIn {
  float4 a;   // residual (o_proj, down) or RoPE (cos, sin) of columns j, j+1 (q, k)
  float4 b;   // RoPE (cos, sin) of columns j+2, j+3 (q, k)
};
__device__ __forceinline__ int qkv_which(const ChainParams& P, int t) {
  const int tq = P.Hd / 128, tk = P.Gd / 128;
  return t < tq ? 0 : t < tq + tk ? 1 : 2;
}

// The gain the tile's epilogue multiplies by (the same for all rows): the
// next norm's (o_proj, down), the head norm's (q, k) or none.
__device__ __forceinline__ float4 tile_gain(const ChainParams& P, int kind, int l, int t) {
  const int lane = threadIdx.x & 31;
  if (kind == PH_O || kind == PH_DN) {
    const float* gn = kind == PH_O ? P.lay[l].g_post : l + 1 < P.nL ? P.lay[l + 1].g_in : P.g_f;
    return __ldg((const float4*)(gn + t * 128) + lane);
  }
  if (kind == PH_QKV && P.qk_norm) {
    const int which = qkv_which(P, t);
    if (which < 2) return __ldg((const float4*)(which == 0 ? P.lay[l].q_norm : P.lay[l].k_norm) + lane);
  }
  return make_float4(1.f, 1.f, 1.f, 1.f);
}

__device__ __forceinline__ RowIn row_in(const ChainParams& P, int kind, int t, int r,
                                        const int* rowpos) {
  const int lane = threadIdx.x & 31;
  RowIn in;
  in.a = in.b = make_float4(0.f, 0.f, 0.f, 0.f);
  if (kind == PH_O || kind == PH_DN) {
    in.a = __ldcg((const float4*)(P.x + (int64_t)r * P.D + t * 128) + lane);
  } else if (kind == PH_QKV && qkv_which(P, t) < 2) {
    const int pos = rowpos[2 * r + 1];
    if (pos >= 0 && pos < P.max_pos) {
      const float4* rp = (const float4*)(P.rope + (int64_t)pos * 64 + ((4 * lane) & 63));
      in.a = __ldg(rp);
      in.b = __ldg(rp + 1);
    }
  }
  return in;
}

__device__ __forceinline__ void row_apply(const ChainParams& P, int kind, int t, int r, float4 v,
                                          float4 g, const RowIn& in, const int* rowpos,
                                          float* rec /* [16][3] of this warp */) {
  const int lane = threadIdx.x & 31;
  if (kind == PH_O || kind == PH_DN) {
    // x += v; x * g for the next norm; the row's sum of squares over the tile
    const float4 nv = make_float4(in.a.x + v.x, in.a.y + v.y, in.a.z + v.z, in.a.w + v.w);
    const int64_t off = (int64_t)r * P.D + t * 128 + 4 * lane;
    *(float4*)(P.x + off) = nv;
    *(float4*)(P.xg + off) = make_float4(nv.x * g.x, nv.y * g.y, nv.z * g.z, nv.w * g.w);
    const float ss = warp_sum(nv.x * nv.x + nv.y * nv.y + nv.z * nv.z + nv.w * nv.w);
    if (lane == 0) P.ssq[(t * CH_ROWS + r) * CH_SSQ] = ss;
  } else if (kind == PH_GU) {
    // columns 0..63: gate rows of the tile, 64..127: up rows
    const float4 u = shfl_xor4(v, 16);
    if (lane < 16) {
      uint2 pk;
      pk.x = pack_bf16(v.x / (1.0f + expf(-v.x)) * u.x, v.y / (1.0f + expf(-v.y)) * u.y);
      pk.y = pack_bf16(v.z / (1.0f + expf(-v.z)) * u.z, v.w / (1.0f + expf(-v.w)) * u.w);
      *(uint2*)(P.a + (int64_t)r * P.F + t * 64 + 4 * lane) = pk;
    }
  } else if (kind == PH_QKV) {
    const int which = qkv_which(P, t);
    const int tq = P.Hd / 128, tk = P.Gd / 128;
    if (which < 2) {
      if (P.qk_norm) {   // per-head RMSNorm over the tile's 128 columns
        const float ss = warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w);
        const float rinv = 1.0f / sqrtf(ss / (float)CH_DH + P.eps);
        v = make_float4(v.x * rinv * g.x, v.y * rinv * g.y, v.z * rinv * g.z, v.w * rinv * g.w);
      }
      const int pos = rowpos[2 * r + 1];
      if (pos < 0 || pos >= P.max_pos) {
        if (lane == 0) atomicOr(P.status, ST_BOUNDS);
        return;
      }
      // rotate-half pairs (j, j + 64): lanes 0-15 hold j, lanes 16-31 j + 64
      const float4 o = shfl_xor4(v, 16);
      const float sg = lane < 16 ? -1.f : 1.f;
      const float4 c0 = in.a, c1 = in.b;   // (cos, sin) of j, j+1 | j+2, j+3
      v = make_float4(v.x * c0.x + sg * o.x * c0.y, v.y * c0.z + sg * o.y * c0.w,
                      v.z * c1.x + sg * o.z * c1.y, v.w * c1.z + sg * o.w * c1.w);
    }
    bf16* dst = which == 0 ? P.q + (int64_t)r * P.Hd + t * CH_DH
                : which == 1 ? P.kb + (int64_t)r * P.Gd + (t - tq) * CH_DH
                             : P.vb + (int64_t)r * P.Gd + (t - tq - tk) * CH_DH;
    uint2 pk;
    pk.x = pack_bf16(v.x, v.y);
    pk.y = pack_bf16(v.z, v.w);
    *(uint2*)(dst + 4 * lane) = pk;
  } else {   // PH_LM: top-2 of the tile's row, folded into this warp's record
    Top2 tt{-INFINITY, 0x7fffffff, -INFINITY};
    const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int n = t * 128 + 4 * lane + k;
      if (n < P.V) tt = top2_merge(tt, Top2{vv[k], n, -INFINITY});
    }
    tt = top2_warp(tt);
    if (lane == 0) {
      Top2 cur{rec[3 * r], __float_as_int(rec[3 * r + 1]), rec[3 * r + 2]};
      cur = top2_merge(cur, tt);
      rec[3 * r] = cur.t1;
      rec[3 * r + 1] = __int_as_float(cur.i1);
      rec[3 * r + 2] = cur.t2;
    }
  }
}

// Row epilogues of the round's projections: the fusion (the row and its sum of squares over the tile) and
// the injection (k: per-head RMSNorm + RoPE; k and v appended to layer li's
// cache at the row's position).  injpos: (sequence, position) per pending row.
__device__ __forceinline__ void row_round(const ChainParams& P, int kind, int t, int r, float4 v,
                                       const int* injpos) {
  const int lane = threadIdx.x & 31;
  if (kind == PH_FUSE) {
    *(float4*)(P.x + (int64_t)r * P.D + t * 128 + 4 * lane) = v;
    const float ss = warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w);
    if (lane == 0) P.ssq[(t * CH_ROWS + r) * CH_SSQ] = ss;
    return;
  }
  const int tk = P.Gd / 128, li = t / (2 * tk), w = (t - li * 2 * tk) / tk;
  const int head = t - li * 2 * tk - w * tk;
  if (w == 0 && P.qk_norm) {
    const float4 g = __ldg((const float4*)P.lay[li].k_norm + lane);
    const float ss = warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w);
    const float rinv = 1.0f / sqrtf(ss / (float)CH_DH + P.eps);
    v = make_float4(v.x * rinv * g.x, v.y * rinv * g.y, v.z * rinv * g.z, v.w * rinv * g.w);
  }
  const int b = injpos[2 * r], pos = injpos[2 * r + 1];
  if (b < 0) return;   // not a pending row of any sequence
  if (pos < 0 || pos >= P.cap || b >= P.kv_batch || (w == 0 && pos >= P.max_pos)) {
    if (lane == 0) atomicOr(P.status, ST_CAPACITY);
    return;
  }
  if (w == 0) {   // rotate-half pairs (j, j + 64): lanes 0-15 hold j, lanes 16-31 j + 64
    const float4* rp = (const float4*)(P.rope + (int64_t)pos * 64 + ((4 * lane) & 63));
    const float4 c0 = __ldg(rp), c1 = __ldg(rp + 1);
    const float4 o = shfl_xor4(v, 16);
    const float sg = lane < 16 ? -1.f : 1.f;
    v = make_float4(v.x * c0.x + sg * o.x * c0.y, v.y * c0.z + sg * o.y * c0.w,
                    v.z * c1.x + sg * o.z * c1.y, v.w * c1.z + sg * o.w * c1.w);
  }
  bf16* dst = const_cast<bf16*>(w == 0 ? P.kc[li] : P.vc[li]) +
              (((int64_t)b * P.G + head) * P.cap + pos) * CH_DH;
  uint2 pk;
  pk.x = pack_bf16(v.x, v.y);
  pk.y = pack_bf16(v.z, v.w);
  *(uint2*)(dst + 4 * lane) = pk;
}

// 1 / rms of every row of the residual from its per-(tile, row) sums of
// squares, into rinv_s (all consumer threads; 8 per row take every 8th tile,
// loads in flight together, then a fixed shuffle tree adds the 8 parts).
__device__ void rinv_rows(const ChainParams& P, float* rinv_s) {
  const int tid = threadIdx.x - 32;
  const int r = tid >> 3, j = tid & 7, nt = P.D / 128;
  float s = 0.f;
  for (int t0 = j; t0 < nt; t0 += 64) {
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int t = t0 + 8 * k;
      v[k] = t < nt ? __ldcg(P.ssq + (t * CH_ROWS + r) * CH_SSQ) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) s += v[k];
  }
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  s += __shfl_xor_sync(0xffffffffu, s, 4);
  named_bar(1, CH_CT);   // the previous readers of rinv_s are done
  if (j == 0) rinv_s[r] = r < P.R ? 1.0f / sqrtf(s / (float)P.D + P.eps) : 0.f;
  named_bar(1, CH_CT);
}

// A normalised operand's unit: round its fp32 (x * g) chunk [16 rows][64 k]
// from the ring stage into the bf16 tile bf16(x * g / rms) at dst (the
// 128-byte swizzled layout of the bf16 loads), one of two buffers at the
// start of the epilogue tile E, which no TMA load writes.  A buffer is
// rewritten two units later, after every warp has passed the barrier of the
// unit between; after a flush (E rewritten and read by the epilogues)
// `sync_first` waits for every warp first.  Every consumer thread takes the
// barriers whatever `ok` says, so the warps stay in step after an abort.
__device__ __forceinline__ void normalise_chunk(const uint8_t* st, uint8_t* dst,
                                                const float* rinv_s, bool ok, bool sync_first) {
  const int tid = threadIdx.x - 32;
  if (sync_first) named_bar(1, CH_CT);
  if (ok) {
    const int c = tid & 15;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float4 f = ((const float4*)st)[tid + h * CH_CT];   // row tid / 16 + 8 h, k 4 c ..
      const int r = (tid >> 4) + 8 * h;
      const float ri = rinv_s[r];
      uint2 pk;
      pk.x = pack_bf16(f.x * ri, f.y * ri);
      pk.y = pack_bf16(f.z * ri, f.w * ri);
      *(uint2*)(dst + r * 128 + (((c >> 1) ^ (r & 7)) << 4) + (c & 1) * 8) = pk;
    }
  }
  named_bar(1, CH_CT);   // the tile is complete before any warp reads it
}

// One projection phase: this CTA's units [u0, u1) of the phase's
// (tile, k-chunk) grid.  A tile whose units this CTA owns entirely is
// finished here (row epilogues); every other tile leaves this CTA's partial
// sum in its slot for the reduce phase.  `ri` is the ring index of the first
// unit.  After a timed-out wait the warps skip the arithmetic but keep every
// barrier.
template <bool RD>
__device__ void gemm_phase(const ChainParams& P, int phase, int kind, int l, int& ri,
                           uint8_t* smem, uint32_t sbase, uint32_t bar_full, uint32_t bar_empty,
                           volatile int* misc, const int* rowpos, float* rinv_s, float* recs) {
  const int tid = threadIdx.x - 32, cw = tid >> 5, lane = threadIdx.x & 31;
  const Geo geo = gemm_geo(P, kind);
  const int cta = blockIdx.x;
  int u0, u1;
  unit_range(P, kind, cta, u0, u1);
  if (u1 <= u0) return;
  float* E = (float*)(smem + CH_OFF_E);
  const int g = lane >> 2, tg = lane & 3;
  const int nrows = rows_of<RD>(P, kind);
  // 1 / rms of every row from the sums of squares the previous phases wrote
  // (these loads overlap the first units' activation loads)
  if (geo.nin) rinv_rows(P, rinv_s);
  float acc[4][4];
  int cur = -1, kbeg = 0, kend = 0;
  bool flushed = false;   // E was written since the last rounded unit

  auto flush = [&](int t) -> void {
    named_bar(1, CH_CT);   // the previous tile's rows have been read out of E
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = cw * 32 + j * 8 + 2 * tg;
      *(float2*)&E[g * CH_EPAD + col] = make_float2(acc[j][0], acc[j][1]);
      *(float2*)&E[(g + 8) * CH_EPAD + col] = make_float2(acc[j][2], acc[j][3]);
    }
    named_bar(1, CH_CT);
    if (kbeg == 0 && kend == geo.kc) {
      // whole tile: finish its rows here (warp cw: rows cw, cw + 4, ...)
      const float4 gt = tile_gain(P, kind, l, t);
      RowIn in[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = cw + 4 * q;
        in[q] = row_in(P, kind, t, r < nrows ? r : 0, rowpos);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = cw + 4 * q;
        if (r >= nrows) continue;
        if (RD && (kind == PH_FUSE || kind == PH_INJ))
          row_round(P, kind, t, r, *(const float4*)&E[r * CH_EPAD + 4 * lane], rowpos);
        else
          row_apply(P, kind, t, r, *(const float4*)&E[r * CH_EPAD + 4 * lane], gt, in[q], rowpos,
                    recs + cw * 48);
      }
    } else {
      const int slot_i = (uint32_t)u0 / (uint32_t)geo.kc == (uint32_t)t ? 0 : 1;
      float4* slot = (float4*)(P.partial + (int64_t)(2 * cta + slot_i) * (CH_ROWS * 128));
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e4 = tid + q * CH_CT, e = e4 * 4;
        slot[e4] = *(const float4*)&E[(e >> 7) * CH_EPAD + (e & 127)];
      }
    }
  };

  int t = u0 / geo.kc, kk = u0 - t * geo.kc - 1;   // advanced at the top of each turn
  for (int u = u0; u < u1; ++u, ++ri) {
    if (++kk == geo.kc) {
      kk = 0;
      ++t;
    }
    if (t != cur) {
      if (cur >= 0) {
        flush(cur);
        flushed = true;
      }
      cur = t;
      kbeg = kk;
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    }
    const int s = ri % CH_STAGES;
    kend = kk + 1;
    bool ok = misc[MS_ABORT] == 0;
    if (ok && !__any_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, (ri / CH_STAGES) & 1))) {
      if (lane == 0) atomicOr(P.status, ST_TIMEOUT);
      misc[MS_ABORT] = 1;
      ok = false;
    }
    if (geo.nin) {
      normalise_chunk(smem + CH_OFF_A + s * CH_AS, smem + CH_OFF_E + (u & 1) * CH_A, rinv_s, ok,
                      flushed);
      flushed = false;
    }
    if (!ok) continue;
    if (DFLASH_CH_EVLOG && tid == 0 && u - u0 < kEvUnits) ev(P, phase, 2 + (u - u0));
    const uint32_t wb = sbase + s * CH_W;
    const uint32_t ab = geo.nin ? sbase + CH_OFF_E + (u & 1) * CH_A : sbase + CH_OFF_A + s * CH_AS;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      uint32_t af[4];
      {
        const int row = lane & 15, ch = 2 * ks + (lane >> 4);
        ldsm_x4(ab + row * 128 + ((ch ^ (row & 7)) << 4), af[0], af[1], af[2], af[3]);
      }
      uint32_t b[4][2];
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        const int row = cw * 32 + pp * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int ch = 2 * ks + ((lane >> 3) & 1);
        ldsm_x4(wb + row * 128 + ((ch ^ (row & 7)) << 4), b[2 * pp][0], b[2 * pp][1],
                b[2 * pp + 1][0], b[2 * pp + 1][1]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) mma_bf16_16816(acc[j], af, b[j][0], b[j][1]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    if (tid == 0) {
      if (DFLASH_CH_EVLOG && u - u0 < kEvUnits) ev(P, phase, 2 + kEvUnits + (u - u0));
      misc[MS_CONSUMED] = ri + 1;
      if (u == u0) trace_max(P, 5, phase);                  // first unit ready and done
      if (u == u0 + (u1 - u0) / 2) trace_max(P, 6, phase);  // half of the units done
    }
  }
  if (P.trace != nullptr && tid == 0)   // last CTA to finish its multiply-adds
    atomicMax(P.trace + 4 * kChainMaxPhases + phase, (unsigned long long)globaltimer());
  flush(cur);
}

// Reduce phase after a projection: one warp per (tile, row) of every tile
// that several CTAs contributed to adds the contributors' partial rows in
// CTA (= k) order, with all loads of a batch (and the epilogue's own inputs)
// in flight together, then runs the row epilogue.
//
// Contributors of tile t (units t*kc .. t*kc + kc - 1): with at least one unit
// per CTA (U >= G) they are the CTAs lo .. hi, each of which holds t in slot 0
// (its first tile) except lo when lo began in an earlier tile (slot 1); with
// fewer units than CTAs every unit has its own owner, holding t in slot 0.
template <bool RD>
__device__ void reduce_phase(const ChainParams& P, int kind, int l, const int* rowpos, float* recs) {
  const int warp = (threadIdx.x - 32) >> 5, lane = threadIdx.x & 31;
  const Geo geo = gemm_geo(P, kind);
  const uint32_t Uu = (uint32_t)geo.n_tiles * geo.kc;
  if (kind == PH_LM && Uu >= 2u * geo.kc * P.grid) {
    // At least two whole tiles' units per CTA: a split tile contains exactly
    // one CTA boundary, so its contributors are CTA c - 1 (slot 1) and CTA c
    // (slot 0).  One warp per (boundary, 4 rows): 8 loads in one batch.
    const int nq = (P.R + 3) / 4;
    const RowIn none{make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    for (int k = blockIdx.x * 4 + warp; k < (P.grid - 1) * nq; k += P.grid * 4) {
      const int c = 1 + k / nq, r0 = (k - (c - 1) * nq) * 4;
      const uint32_t fu = (uint32_t)c * Uu / (uint32_t)P.grid;
      if (fu % geo.kc == 0) continue;   // boundary between tiles: nothing split
      const int t = fu / geo.kc;
      const float* pa = P.partial + (int64_t)(2 * (c - 1) + 1) * (CH_ROWS * 128);
      const float* pb = P.partial + (int64_t)(2 * c) * (CH_ROWS * 128);
      float4 va[4], vb[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = min(r0 + q, P.R - 1);
        va[q] = __ldcg((const float4*)(pa + r * 128) + lane);
        vb[q] = __ldcg((const float4*)(pb + r * 128) + lane);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = r0 + q;
        if (r >= P.R) break;
        const float4 sum = make_float4(0.f + va[q].x + vb[q].x, 0.f + va[q].y + vb[q].y,
                                       0.f + va[q].z + vb[q].z, 0.f + va[q].w + vb[q].w);
        row_apply(P, kind, t, r, sum, make_float4(1.f, 1.f, 1.f, 1.f), none, rowpos,
                  recs + warp * 48);
      }
    }
    return;
  }
  if (kind == PH_GU && Uu >= (uint32_t)P.grid && 3u * (Uu / P.grid) >= geo.kc) {
    // gate/up (an epilogue that reads nothing per row) with at least kc / 3
    // units per CTA: a split tile has at most 3 contributors (CTAs lo .. hi,
    // lo in slot 1 when it began in an earlier tile).  One warp per (tile,
    // 4 rows): all of a task's loads in one batch, one task per warp.
    constexpr int CB = 3;
    const uint32_t G = P.grid;
    auto owner = [&](uint32_t u) { return (int)(((u + 1) * G + Uu - 1) / Uu) - 1; };
    const int nq = (P.R + 3) / 4;
    const RowIn none{make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    for (int k = blockIdx.x * 4 + warp; k < geo.n_tiles * nq; k += P.grid * 4) {
      const int t = k / nq, r0 = (k - t * nq) * 4;
      const int lo = owner((uint32_t)t * geo.kc), hi = owner((uint32_t)t * geo.kc + geo.kc - 1);
      if (lo == hi) continue;   // finished by its only owner
      const int n = hi - lo + 1;
      const bool lo1 = (uint32_t)lo * Uu / G < (uint32_t)t * geo.kc;
      float4 v[CB][4];
#pragma unroll
      for (int j = 0; j < CB; ++j) {
        const float* pj = P.partial + (int64_t)(2 * (lo + j) + (j == 0 && lo1 ? 1 : 0)) * (CH_ROWS * 128);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = min(r0 + q, P.R - 1);
          v[j][q] = j < n ? __ldcg((const float4*)(pj + r * 128) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = r0 + q;
        if (r >= P.R) break;
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < CB; ++j) {
          sum.x += v[j][q].x;
          sum.y += v[j][q].y;
          sum.z += v[j][q].z;
          sum.w += v[j][q].w;
        }
        row_apply(P, kind, t, r, sum, make_float4(1.f, 1.f, 1.f, 1.f), none, rowpos,
                  recs + warp * 48);
      }
    }
    return;
  }
  const uint32_t U = (uint32_t)geo.n_tiles * geo.kc, G = P.grid, kc = geo.kc;
  const int R = rows_of<RD>(P, kind), ntask = geo.n_tiles * R;
  const bool dense = U >= G;
  auto owner = [&](uint32_t u) { return (int)(((u + 1) * G + U - 1) / U) - 1; };
  constexpr int RB = 12;   // contributors per batch
  const int W = P.grid * 4, k_first = blockIdx.x * 4 + warp;
  for (int k = k_first; k < ntask; k += W) {
    const int t = k / R, r = k - t * R;
    const int lo = owner((uint32_t)t * kc), hi = owner((uint32_t)t * kc + kc - 1);
    if (lo == hi) continue;   // finished by its only owner
    const int n = dense ? hi - lo + 1 : (int)kc;
    const bool lo_slot1 = dense && (uint32_t)lo * U / G < (uint32_t)t * kc;
    const float4 gt = tile_gain(P, kind, l, t);
    const RowIn in = row_in(P, kind, t, r, rowpos);
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < n; j0 += RB) {
      float4 v[RB];
#pragma unroll
      for (int j = 0; j < RB; ++j) {
        v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j0 + j < n) {
          const int c = dense ? lo + j0 + j : owner((uint32_t)t * kc + j0 + j);
          const int slot = (dense && j0 + j == 0 && lo_slot1) ? 1 : 0;
          v[j] = __ldcg((const float4*)(P.partial + (int64_t)(2 * c + slot) * (CH_ROWS * 128) +
                                        r * 128) + lane);
        }
      }
#pragma unroll
      for (int j = 0; j < RB; ++j) {
        sum.x += v[j].x;
        sum.y += v[j].y;
        sum.z += v[j].z;
        sum.w += v[j].w;
      }
    }
    if (RD && (kind == PH_FUSE || kind == PH_INJ))
      row_round(P, kind, t, r, sum, rowpos);
    else
      row_apply(P, kind, t, r, sum, gt, in, rowpos, recs + warp * 48);
  }
}

// End of the LM head's reduce phase: each CTA publishes one top-2 record per
// row (over the vocabulary tiles it finished, from its four warps' records).
__device__ void lm_publish(const ChainParams& P, const float* recs) {
  const int tid = threadIdx.x - 32;
  named_bar(1, CH_CT);
  if (tid < P.R) {
    Top2 m{-INFINITY, 0x7fffffff, -INFINITY};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float* rc = recs + w * 48 + 3 * tid;
      m = top2_merge(m, Top2{rc[0], __float_as_int(rc[1]), rc[2]});
    }
    P.amx[(int64_t)blockIdx.x * P.R + tid] = make_float4(m.t1, __int_as_float(m.i1), m.t2, 0.f);
  }
}

// Final merge (after a grid barrier): one warp per row merges the grid's
// records (top-2 merging is order-free, so the result does not depend on
// which CTA finished which tile) and writes the id and the gap.
__device__ void lm_merge(const ChainParams& P) {
  const int warp = (threadIdx.x - 32) >> 5, lane = threadIdx.x & 31;
  const int R = P.R;
  for (int r = blockIdx.x * 4 + warp; r < R; r += P.grid * 4) {
    const int b = r / P.B, i = r - b * P.B;
    if (i == 0) {
      if (lane == 0) P.ids[(int64_t)b * P.B] = P.anchor[b];
      continue;
    }
    Top2 tt{-INFINITY, 0x7fffffff, -INFINITY};
    for (int c0 = 0; c0 < P.grid; c0 += 32 * 12) {
      float4 v[12];
#pragma unroll
      for (int q = 0; q < 12; ++q) {
        const int c = c0 + lane + 32 * q;
        v[q] = c < P.grid ? __ldcg(&P.amx[(int64_t)c * R + r])
                          : make_float4(-INFINITY, __int_as_float(0x7fffffff), -INFINITY, 0.f);
      }
#pragma unroll
      for (int q = 0; q < 12; ++q) tt = top2_merge(tt, Top2{v[q].x, __float_as_int(v[q].y), v[q].z});
    }
    tt = top2_warp(tt);
    if (lane == 0) {
      float g = tt.t1 - tt.t2;
      P.ids[(int64_t)b * P.B + i] = argmax_id(tt.i1, g, P.status);
      if (P.gap) P.gap[(int64_t)b * (P.B - 1) + i - 1] = g;
    }
  }
}

// ---- consumers: attention ----------------------------------------------------------
// Work items: for each sequence b, the keys [0, len_b + B) in 32-key
// sub-chunks, `chunk` sub-chunks per item; items ordered (b, g, run).
struct Items {
  int chunk, total;
  int nsub[CH_MAXB], runs[CH_MAXB], base[CH_MAXB], L[CH_MAXB];
};

template <bool RD>
__device__ void make_items(const ChainParams& P, Items* it) {
  int U = 0;
  for (int b = 0; b < P.batch; ++b) {
    int L = P.len[b] + (RD && P.pre ? P.nrow[b] : 0);   // a round's appended rows count
    if (L < 0 || L > P.cap) {
      atomicOr(P.status, ST_BOUNDS);
      L = L < 0 ? 0 : P.cap;
    }
    it->L[b] = L;
    it->nsub[b] = (L + P.B + CH_AK - 1) / CH_AK;
    U += P.G * it->nsub[b];
  }
  const int chunk = max(1, (U + P.grid - 1) / P.grid);
  int n = 0;
  for (int b = 0; b < P.batch; ++b) {
    it->runs[b] = (it->nsub[b] + chunk - 1) / chunk;
    it->base[b] = n;
    n += P.G * it->runs[b];
  }
  it->chunk = chunk;
  it->total = n;
}

__device__ __forceinline__ uint32_t tswz(int row, int chunk) {
  return (uint32_t)(row * (CH_DH * 2) + ((chunk ^ (row & 7)) << 4));
}

struct ItemGeo {
  int b, g, L, k_begin, k_end;
};
__device__ __forceinline__ ItemGeo item_geo(const ChainParams& P, const Items* it, int j) {
  ItemGeo q;
  q.b = 0;
  while (q.b + 1 < P.batch && j >= it->base[q.b + 1]) ++q.b;
  const int jj = j - it->base[q.b];
  q.g = jj / it->runs[q.b];
  const int run = jj - q.g * it->runs[q.b];
  q.L = it->L[q.b];
  q.k_begin = run * it->chunk * CH_AK;
  q.k_end = min(q.L + P.B, q.k_begin + it->chunk * CH_AK);
  return q;
}

__device__ void attention_phase(const ChainParams& P, int phase, int l, const Items* it, uint8_t* smem,
                                const int* rowpos) {
  const int tid = threadIdx.x - 32, warp = tid >> 5, lane = threadIdx.x & 31;
  const uint32_t sQ = smem_u32(smem + CH_OFF_ATT);
  const uint32_t sK0 = sQ + CH_ATT_Q, sV0 = sK0 + 2 * CH_ATT_KV;
  const int QM = P.B * P.rep;
  const int gq = lane >> 2, tg = lane & 3;
  const bool active = warp * 16 < QM;
  const int total = min(it->total, P.n_items_max);
  for (int j = blockIdx.x; j < total; j += P.grid) {
    const ItemGeo ig = item_geo(P, it, j);
    const int b = ig.b, g = ig.g, L = ig.L, k_begin = ig.k_begin, k_end = ig.k_end;
    const int nsub = (k_end - k_begin + CH_AK - 1) / CH_AK;
    // a causal or windowed layer (CTA-uniform): each query row sees keys
    // [klo, khi) only; the other layers run the unmasked code as it is
    const bool masked = ((P.causal_layers | P.window_layers) >> l) & 1;
    const bf16* kcb = P.kc[l] + ((int64_t)b * P.G + g) * P.cap * CH_DH;
    const bf16* vcb = P.vc[l] + ((int64_t)b * P.G + g) * P.cap * CH_DH;
    const bf16* kbb = P.kb + (int64_t)b * P.B * P.Gd + (int64_t)g * CH_DH;
    const bf16* vbb = P.vb + (int64_t)b * P.B * P.Gd + (int64_t)g * CH_DH;
    named_bar(1, CH_CT);   // the previous item is done with the buffers
    // Q rows: row r = head hh of the group, block row i (r = hh * B + i)
    for (int e = tid; e < 64 * 16; e += CH_CT) {
      const int r = e >> 4, c = e & 15;
      const bool ok = r < QM;
      const int hh = ok ? r / P.B : 0, i = ok ? r - hh * P.B : 0;
      const bf16* src = P.q + (int64_t)(b * P.B + i) * P.Hd + (int64_t)(g * P.rep + hh) * CH_DH + c * 8;
      cp_async16(sQ + tswz(r, c), ok ? src : P.q, ok);
    }
    auto load_kv = [&](int k0, int stage) {
      const uint32_t dk = sK0 + stage * CH_ATT_KV, dv = sV0 + stage * CH_ATT_KV;
      for (int e = tid; e < CH_AK * 16; e += CH_CT) {
        const int r = e >> 4, c = e & 15, jk = k0 + r;
        const bool ok = jk < k_end;
        const bf16 *ks, *vs;
        if (jk < L) {
          ks = kcb + (int64_t)jk * CH_DH + c * 8;
          vs = vcb + (int64_t)jk * CH_DH + c * 8;
        } else {
          const int jb = ok ? jk - L : 0;
          ks = kbb + (int64_t)jb * P.Gd + c * 8;
          vs = vbb + (int64_t)jb * P.Gd + c * 8;
        }
        cp_async16(dk + tswz(r, c), ok ? ks : kcb, ok);
        cp_async16(dv + tswz(r, c), ok ? vs : vcb, ok);
      }
    };
    load_kv(k_begin, 0);
    cp_async_commit();
    float acc[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    for (int sc = 0; sc < nsub; ++sc) {
      const int stage = sc & 1;
      if (sc + 1 < nsub) load_kv(k_begin + (sc + 1) * CH_AK, stage ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
      named_bar(1, CH_CT);
      if (sc == 0 && tid == 0) trace_max(P, 5, phase);   // first K/V sub-chunk in
      if (active) {
        const uint32_t sK = sK0 + stage * CH_ATT_KV, sV = sV0 + stage * CH_ATT_KV;
        const int kbase = k_begin + sc * CH_AK;
        float s[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t qa[4];   // Q fragments are re-read from shared memory (registers are scarce)
          {
            const int row = warp * 16 + (lane & 15), ch = 2 * ks + (lane >> 4);
            ldsm_x4(sQ + tswz(row, ch), qa[0], qa[1], qa[2], qa[3]);
          }
#pragma unroll
          for (int pp = 0; pp < 2; ++pp) {
            const int row = pp * 16 + (lane & 7) + ((lane >> 4) << 3);
            const int ch = 2 * ks + ((lane >> 3) & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(sK + tswz(row, ch), b0, b1, b2, b3);
            mma_bf16_16816(s[2 * pp], qa, b0, b1);
            mma_bf16_16816(s[2 * pp + 1], qa, b2, b3);
          }
        }
        float mnew[2] = {mrow[0], mrow[1]};
        if (!masked) {
#pragma unroll
          for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int key = kbase + n * 8 + 2 * tg + (q & 1);
              s[n][q] = key < k_end ? s[n][q] * P.scale_log2 : -INFINITY;
              mnew[q >> 1] = fmaxf(mnew[q >> 1], s[n][q]);
            }
        } else {
          // this thread's rows r (= hh * B + i) and r + 8: block row i at
          // position rowpos; causal keeps keys up to it, a window of W the
          // last W positions
          const int win = ((P.window_layers >> l) & 1) ? P.window : 0;
          const bool causal = (P.causal_layers >> l) & 1;
          int klo[2], khi[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int r = warp * 16 + gq + 8 * h;
            const int pq = rowpos[2 * (b * P.B + (r < QM ? r % P.B : 0)) + 1];
            klo[h] = win > 0 ? max(0, pq - win + 1) : 0;
            khi[h] = causal ? pq + 1 : k_end;
          }
#pragma unroll
          for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int key = kbase + n * 8 + 2 * tg + (q & 1);
              const bool vis = key < k_end && key >= klo[q >> 1] && key < khi[q >> 1];
              s[n][q] = vis ? s[n][q] * P.scale_log2 : -INFINITY;
              mnew[q >> 1] = fmaxf(mnew[q >> 1], s[n][q]);
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mnew[h] = fmaxf(mnew[h], __shfl_xor_sync(0xffffffffu, mnew[h], 1));
          mnew[h] = fmaxf(mnew[h], __shfl_xor_sync(0xffffffffu, mnew[h], 2));
        }
        float alpha[2], lsum[2] = {0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h) alpha[h] = mrow[h] == -INFINITY ? 0.f : exp2f(mrow[h] - mnew[h]);
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            // a masked row may see no key of this item yet: weight 0
            const float e = masked && mnew[q >> 1] == -INFINITY ? 0.f : exp2f(s[n][q] - mnew[q >> 1]);
            s[n][q] = e;
            lsum[q >> 1] += e;
          }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          lrow[h] = lrow[h] * alpha[h] + lsum[h];
          mrow[h] = mnew[h];
        }
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          acc[n][0] *= alpha[0];
          acc[n][1] *= alpha[0];
          acc[n][2] *= alpha[1];
          acc[n][3] *= alpha[1];
        }
        // O += P V with P rounded to bf16 (plus its bf16 remainder when DFLASH_CH_PLO)
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const float* s0 = s[2 * kk];
          const float* s1 = s[2 * kk + 1];
          const float v[8] = {s0[0], s0[1], s0[2], s0[3], s1[0], s1[1], s1[2], s1[3]};
          float hi[8], lo[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            hi[q] = __bfloat162float(__float2bfloat16_rn(v[q]));
            lo[q] = v[q] - hi[q];
          }
          const uint32_t ph[4] = {pack_bf16(hi[0], hi[1]), pack_bf16(hi[2], hi[3]),
                                  pack_bf16(hi[4], hi[5]), pack_bf16(hi[6], hi[7])};
          const uint32_t pl[4] = {pack_bf16(lo[0], lo[1]), pack_bf16(lo[2], lo[3]),
                                  pack_bf16(lo[4], lo[5]), pack_bf16(lo[6], lo[7])};
#pragma unroll
          for (int np = 0; np < 8; ++np) {
            const int row = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
            const int ch = np * 2 + (lane >> 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(sV + tswz(row, ch), b0, b1, b2, b3);
            mma_bf16_16816(acc[2 * np], ph, b0, b1);
            mma_bf16_16816(acc[2 * np + 1], ph, b2, b3);
            if (DFLASH_CH_PLO) {
              mma_bf16_16816(acc[2 * np], pl, b0, b1);
              mma_bf16_16816(acc[2 * np + 1], pl, b2, b3);
            }
          }
        }
      }
      named_bar(1, CH_CT);   // stage buffers free for the load two steps ahead
    }
    cp_async_wait<0>();
    if (tid == 0) trace_max(P, 6, phase);   // item's arithmetic done
    if (active) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 1);
        lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 2);
      }
      float* part = P.apart + (int64_t)j * 64 * CH_DP;
      const int r0 = warp * 16 + gq, r1 = r0 + 8;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        const int col = n * 8 + 2 * tg;
        *(float2*)&part[r0 * CH_DP + 4 + col] = make_float2(acc[n][0], acc[n][1]);
        *(float2*)&part[r1 * CH_DP + 4 + col] = make_float2(acc[n][2], acc[n][3]);
      }
      if (tg == 0) {
        part[r0 * CH_DP] = mrow[0];
        part[r0 * CH_DP + 1] = lrow[0];
        part[r1 * CH_DP] = mrow[1];
        part[r1 * CH_DP + 1] = lrow[1];
      }
    }
    if (tid == 0) trace_max(P, 7, phase);   // partial written (issued)
  }
}

// Combine: two warps per (sequence, kv head, query row), each owning 64 of
// the row's 128 output columns (two per lane).  The runs' (max, sum) pairs
// come in one batch of loads, the runs' outputs in batches of 32 runs; the
// runs are added in run order.
__device__ void combine_phase(const ChainParams& P, int phase, const Items* it) {
  const int tid = threadIdx.x - 32, warp = tid >> 5, lane = threadIdx.x & 31;
  const int QM = P.B * P.rep;
  const int ntask = 2 * P.batch * P.G * QM;
  const int64_t stride = (int64_t)64 * CH_DP;
  for (int w = blockIdx.x * 4 + warp; w < ntask; w += P.grid * 4) {
    const int half = w & 1, row = w >> 1;
    const int b = row / (P.G * QM), rem = row - b * (P.G * QM);
    const int g = rem / QM, r = rem - g * QM;
    const int runs = it->runs[b];
    const int j0 = it->base[b] + g * runs;
    if (j0 + runs > P.n_items_max) continue;
    const float* base = P.apart + ((int64_t)j0 * 64 + r) * CH_DP;
    // (max, sum) of runs lane and lane + 32 stay in registers (at most 64
    // runs); longer lists re-read theirs per group of 32
    float2 ml0 = make_float2(-INFINITY, 0.f), ml1 = make_float2(-INFINITY, 0.f);
    if (lane < runs) ml0 = __ldcg((const float2*)(base + lane * stride));
    if (lane + 32 < runs) ml1 = __ldcg((const float2*)(base + (lane + 32) * stride));
    float M = fmaxf(ml0.x, ml1.x);
    for (int s0 = 64; s0 < runs; s0 += 32)
      if (s0 + lane < runs) M = fmaxf(M, __ldcg(base + (s0 + lane) * stride));
    M = warp_max(M);
    const float w0 = ml0.x == -INFINITY ? 0.f : exp2f(ml0.x - M);
    const float w1 = ml1.x == -INFINITY ? 0.f : exp2f(ml1.x - M);
    float lt = ml0.y * w0 + ml1.y * w1;
    float2 o = make_float2(0.f, 0.f);
    for (int s0 = 0; s0 < runs; s0 += 32) {
      float wl = s0 == 0 ? w0 : w1;
      if (s0 >= 64) {
        const float2 ml = s0 + lane < runs ? __ldcg((const float2*)(base + (s0 + lane) * stride))
                                           : make_float2(-INFINITY, 0.f);
        wl = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
        lt += ml.y * wl;
      }
      float2 v[32];
#pragma unroll
      for (int k = 0; k < 32; ++k)
        v[k] = s0 + k < runs ? __ldcg((const float2*)(base + (s0 + k) * stride + 4 + half * 64) + lane)
                             : make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float wk = __shfl_sync(0xffffffffu, wl, k);
        o.x += v[k].x * wk;
        o.y += v[k].y * wk;
      }
    }
    lt = warp_sum(lt);
    if (lane == 0) trace_max(P, 5, phase);   // weights and outputs in
    const float iv = 1.0f / lt;
    const int hh = r / P.B, i = r - hh * P.B;
    bf16* dst = P.o + (int64_t)(b * P.B + i) * P.Hd + (int64_t)(g * P.rep + hh) * CH_DH +
                half * 64 + 2 * lane;
    *(uint32_t*)dst = pack_bf16(o.x * iv, o.y * iv);
  }
}

// The round's fused context feature: each pending row of the projection
// (fp32 in x) through RMSNorm with gain g_c, H_t = bf16(y / rms(y) * g_c);
// one warp per (row, 128-column tile).  CTA 0 then advances the cache
// lengths by the appended rows (every CTA read them before its first phase).
__device__ void fnorm_phase(const ChainParams& P) {
  const int tid = threadIdx.x - 32, warp = tid >> 5, lane = threadIdx.x & 31;
  const int tiles = P.D / 128;
  for (int w = blockIdx.x * 4 + warp; w < P.n_in * tiles; w += P.grid * 4) {
    const int r = w / tiles, t = w - r * tiles;
    float ss = 0.f;
    for (int tt = lane; tt < tiles; tt += 32) ss += __ldcg(P.ssq + (tt * CH_ROWS + r) * CH_SSQ);
    const float4 y = __ldcg((const float4*)(P.x + (int64_t)r * P.D + t * 128) + lane);
    const float4 g = __ldg((const float4*)(P.g_c + t * 128) + lane);
    const float rinv = 1.0f / sqrtf(warp_sum(ss) / (float)P.D + P.eps);
    uint2 pk;
    pk.x = pack_bf16(y.x * rinv * g.x, y.y * rinv * g.y);
    pk.y = pack_bf16(y.z * rinv * g.z, y.w * rinv * g.w);
    *((uint2*)(P.ht + (int64_t)r * P.D + t * 128) + lane) = pk;
  }
  if (blockIdx.x == 0 && tid < P.batch) P.len[tid] += P.nrow[tid];
}

// Embedding of the block rows (anchor, then mask tokens) into the fp32
// residual, with the per-(tile, row) sums of squares of the first norm.
__device__ void embed_phase(const ChainParams& P) {
  const int tid = threadIdx.x - 32, warp = tid >> 5, lane = threadIdx.x & 31;
  const int tiles = P.D / 128;
  for (int w = blockIdx.x * 4 + warp; w < P.R * tiles; w += P.grid * 4) {
    const int r = w / tiles, t = w - r * tiles;
    const int b = r / P.B, i = r - b * P.B;
    const int id = i == 0 ? P.anchor[b] : P.mask_id;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (id < 0 || id >= P.V) {
      if (lane == 0) atomicOr(P.status, ST_BOUNDS);
    } else {
      const uint2 raw = __ldg((const uint2*)(P.embed + (int64_t)id * P.D + t * 128) + lane);
      const __nv_bfloat162 e0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
      const __nv_bfloat162 e1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
      v = make_float4(__low2float(e0) * P.embed_scale, __high2float(e0) * P.embed_scale,
                      __low2float(e1) * P.embed_scale, __high2float(e1) * P.embed_scale);
    }
    *((float4*)(P.x + (int64_t)r * P.D + t * 128) + lane) = v;
    const float4 g4 = __ldg((const float4*)(P.lay[0].g_in + t * 128) + lane);
    *((float4*)(P.xg + (int64_t)r * P.D + t * 128) + lane) =
        make_float4(v.x * g4.x, v.y * g4.y, v.z * g4.z, v.w * g4.w);
    const float ss = warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w);
    if (lane == 0) P.ssq[(t * CH_ROWS + r) * CH_SSQ] = ss;
  }
}

template <bool RD>
__global__ void __launch_bounds__(CH_THREADS, 2) chain_kernel(const __grid_constant__ ChainParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + CH_OFF_BAR, bar_empty = bar_full + 8 * CH_STAGES;
  volatile int* misc = (volatile int*)(smem + CH_OFF_MISC);
  int* rowpos = (int*)(smem + CH_OFF_MISC) + 16;
  float* rinv_s = (float*)(smem + CH_OFF_MISC) + 48;
  Items* items = (Items*)((int*)(smem + CH_OFF_MISC) + 64);
  float* recs = (float*)(smem + CH_OFF_MISC) + 192;
  int* injpos = (int*)(smem + CH_OFF_MISC) + 384;
  static_assert(64 * 4 + sizeof(Items) <= 192 * 4 && (192 + 4 * 48) * 4 <= 384 * 4 &&
                    (384 + 2 * CH_ROWS) * 4 <= CH_MISC_BYTES, "misc area");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < CH_STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 4);
    }
    misc[MS_ABORT] = misc[MS_LAST] = misc[MS_ISSUED] = misc[MS_CONSUMED] = misc[MS_GO] = 0;
    misc[MS_ATT_DONE] = 0;
    fence_barrier_init();
  }
  if (threadIdx.x == 32) make_items<RD>(P, items);
  if (threadIdx.x >= 32 && threadIdx.x < 32 + CH_ROWS) {
    const int r = threadIdx.x - 32;
    int b = -1, pos = -1;
    if (r < P.R) {
      b = r / P.B;
      pos = P.len[b] + (RD && P.pre ? P.nrow[b] : 0) + (r - b * P.B);
    }
    rowpos[2 * r] = b;
    rowpos[2 * r + 1] = pos;
  }
  if (RD && threadIdx.x >= 64 && threadIdx.x < 64 + CH_ROWS) {
    // a round's pending rows: the sequence whose row range holds the row,
    // and the cache position it is appended at
    const int r = threadIdx.x - 64;
    int b = -1, pos = -1;
    for (int s = 0; P.pre && r < P.n_in && s < P.batch; ++s) {
      const int r0 = P.row0[s], n = P.nrow[s];
      if (r >= r0 && r < r0 + n) {
        b = s;
        pos = P.len[s] + (r - r0);
        break;
      }
    }
    injpos[2 * r] = b;
    injpos[2 * r + 1] = pos;
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) producer<RD>(P, sbase, bar_full, bar_empty, misc);
    __syncwarp();
  } else if (warp == 5) {
    // no work (see CH_THREADS)
  } else {
    const int tid = threadIdx.x - 32;
    int ri = 0;
    for (int p = 0; p < P.n_phases; ++p) {
      if (tid == 0) {
        bool go = misc[MS_ABORT] == 0;
        if (go && !grid_wait(P, p * P.grid)) {
          misc[MS_ABORT] = 1;
          go = false;
        }
        misc[MS_GO] = go;

      }
      named_bar(1, CH_CT);
      if (!misc[MS_GO]) break;
      if (P.trace != nullptr && tid == 0) {
        const unsigned long long now = globaltimer();
        ev(P, p, 0);
        atomicMin(P.trace + p, now);                          // first CTA to start
        atomicMax(P.trace + kChainMaxPhases + p, now);        // last CTA to start
      }
      int l;
      const int kind = phase_kind<RD>(P, p, l);
      if (kind == PH_EMBED) {
        embed_phase(P);
      } else if (kind == PH_ATT) {
        attention_phase(P, p, l, items, smem, rowpos);
        named_bar(1, CH_CT);   // every warp is done with the ring memory
        if (tid == 0) misc[MS_ATT_DONE] = l + 1;
      } else if (kind == PH_CMB) {
        combine_phase(P, p, items);
      } else if (RD && kind == PH_FNORM) {
        fnorm_phase(P);
      } else if (kind == PH_RED) {
        int lp;
        const int pk = phase_kind<RD>(P, p - 1, lp);
        reduce_phase<RD>(P, pk, lp, RD && pk == PH_INJ ? injpos : rowpos, recs);
        if (pk == PH_LM) lm_publish(P, recs);
      } else if (kind == PH_LMFIN) {
        lm_merge(P);
      } else {
        if (kind == PH_LM) {
          for (int e = tid; e < 4 * CH_ROWS; e += CH_CT) {
            recs[3 * e] = -INFINITY;
            recs[3 * e + 1] = __int_as_float(0x7fffffff);
            recs[3 * e + 2] = -INFINITY;
          }
          named_bar(1, CH_CT);
        }
        gemm_phase<RD>(P, p, kind, l, ri, smem, sbase, bar_full, bar_empty, misc,
                       RD && kind == PH_INJ ? injpos : rowpos, rinv_s, recs);
      }
      named_bar(1, CH_CT);
      if (tid == 0) {
        red_release_gpu_add(P.counters + kMaxTiles + 1, 1);
        if (P.trace != nullptr) {
          const unsigned long long now = globaltimer();
          ev(P, p, 1);
          atomicMin(P.trace + 2 * kChainMaxPhases + p, now);  // first CTA to finish
          atomicMax(P.trace + 3 * kChainMaxPhases + p, now);  // last CTA to finish
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (misc[MS_ABORT]) {
      // wait (bounded) for weight / activation loads that were issued but not
      // consumed, so no TMA write lands after the CTA has left
      const int hi = misc[MS_ISSUED];
      for (int i = misc[MS_CONSUMED]; i < hi; ++i)
        if (!mbar_wait(bar_full + 8 * (i % CH_STAGES), (i / CH_STAGES) & 1, 20000000ull)) break;
    } else if (blockIdx.x == 0 && grid_wait(P, P.n_phases * P.grid)) {
      // every CTA has passed its last phase (and polls no more): the barrier
      // counter starts the next launch from zero
      P.counters[kMaxTiles + 1] = 0;
    }
  }
}

// ---------------------------------------------------------------------------
static int g_chain_occ = -1;

int chain_grid(const dflash_handle* h) {
  if (g_chain_occ < 0) {
    int occ = 0;
    // both variants (the block alone, and a round before it) share the
    // launch shape; the grid is what both can keep resident
    int occ1 = 0;
    if (cudaFuncSetAttribute(chain_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             CH_SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(chain_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             CH_SMEM) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, chain_kernel<false>, CH_THREADS,
                                                      CH_SMEM) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ1, chain_kernel<true>, CH_THREADS,
                                                      CH_SMEM) != cudaSuccess)
      occ = occ1 = 0;
    g_chain_occ = std::min(std::min(occ, occ1), 2);
  }
  return g_chain_occ * h->num_sms;
}

size_t chain_apart_bytes(const dflash_handle* h, int batch) {
  const int grid = std::max(chain_grid(h), 2 * h->num_sms);
  return (size_t)(grid + std::max(batch, 1) * h->cfg.n_kv_heads) * 64 * CH_DP * sizeof(float) + 256;
}

bool chain_ok(const dflash_handle* h, int batch, int B) {
  const dflash_config& c = h->cfg;
  const int64_t R = (int64_t)batch * B;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!al16(h->w.g_f)) return false;   // gains are read as float4 in the epilogues
  if (c.conv_group > 0) return false;   // conv modules run in the per-projection path
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash_layer_weights& L = h->w.layers[l];
    if (!al16(L.g_in) || !al16(L.g_post)) return false;
    if (c.qk_norm && (!al16(L.q_norm) || !al16(L.k_norm))) return false;
  }
  return h->have_maps && h->d_wmaps != nullptr && c.dtype == DFLASH_BF16 && c.head_dim == CH_DH &&
         R >= 1 && R <= CH_ROWS && batch <= CH_MAXB && B * (c.n_heads / c.n_kv_heads) <= 64 &&
         c.hidden % 128 == 0 && c.ffn % 64 == 0 && (c.vocab + 127) / 128 <= kMaxTiles &&
         chain_grid(h) > 0;
}

int draft_chain(dflash_handle* h, cudaStream_t s, const ChainArgs& A) {
  const dflash_config& c = h->cfg;
  const int R = A.batch * A.B;
  const int D = c.hidden, Hd = c.n_heads * c.head_dim, Gd = c.n_kv_heads * c.head_dim, F = c.ffn;
  ChainParams P;
  memset(&P, 0, sizeof(P));
  if (!make_tmap_2d(&P.map_xg, A.xg, D, R, (uint64_t)D * 4, 64, 16, DFLASH_F32, false) ||
      !make_tmap_2d(&P.map_o, A.o, Hd, R, (uint64_t)Hd * 2, 64, 16) ||
      !make_tmap_2d(&P.map_a, A.a, F, R, (uint64_t)F * 2, 64, 16))
    return DFLASH_ERR_CUDA;
  if (A.n_in > 0) {
    // the round's phases: the pending features and H_t as TMA sources
    if (A.n_in > CH_ROWS || !A.hidden || !A.row0 || !A.nrow || !A.ht || !h->w.g_c ||
        !h->have_wc_map)
      return DFLASH_ERR_INVALID_ARG;
    for (int i = 0; i < c.n_pick; ++i)
      if (!make_tmap_2d(&P.map_hid[i], A.hidden[i], D, A.n_in, (uint64_t)D * 2, 64, 16))
        return DFLASH_ERR_CUDA;
    if (!make_tmap_2d(&P.map_ht, A.ht, D, A.n_in, (uint64_t)D * 2, 64, 16)) return DFLASH_ERR_CUDA;
    P.pre = kRoundPhases;
    P.n_in = A.n_in;
    P.n_pick = c.n_pick;
    P.row0 = A.row0;
    P.nrow = A.nrow;
    P.ht = (bf16*)A.ht;
    P.g_c = h->w.g_c;
  }
  P.kv_batch = A.kv->batch_cap;
  P.wmaps = h->d_wmaps;
  for (int l = 0; l < c.n_layers; ++l) {
    P.kc[l] = (const bf16*)A.kv->k[l];
    P.vc[l] = (const bf16*)A.kv->v[l];
    const dflash_layer_weights& L = h->w.layers[l];
    P.lay[l] = ChainLayer{L.g_in, L.g_post, L.q_norm, L.k_norm};
  }
  P.embed = (const bf16*)h->w.embed;
  P.g_f = h->w.g_f;
  P.anchor = A.anchor;
  P.len = A.kv->len;   // advanced in place by a round
  P.ids = A.ids;
  P.gap = A.gap;
  P.x = A.x;
  P.xg = A.xg;
  P.q = (bf16*)A.q;
  P.kb = (bf16*)A.kb;
  P.vb = (bf16*)A.vb;
  P.o = (bf16*)A.o;
  P.a = (bf16*)A.a;
  P.ssq = A.ssq;
  P.partial = A.partial;
  P.apart = A.apart;
  P.amx = A.amx;
  P.counters = h->d_counters;
  P.status = h->d_status;
  P.rope = h->d_rope;
  P.max_pos = c.max_pos;
  P.R = R;
  P.batch = A.batch;
  P.B = A.B;
  P.D = D;
  P.Hd = Hd;
  P.Gd = Gd;
  P.F = F;
  P.V = c.vocab;
  P.G = c.n_kv_heads;
  P.rep = c.n_heads / c.n_kv_heads;
  P.nL = c.n_layers;
  P.cap = A.kv->cap;
  P.mask_id = c.mask_token_id;
  P.qk_norm = c.qk_norm;
  P.grid = chain_grid(h);
  if (h->d_trace != nullptr) {
    // minima start from all-ones, maxima from zero
    const size_t col = kChainMaxPhases * sizeof(unsigned long long);
    if (cudaMemsetAsync(h->d_trace, 0xff, col, s) ||
        cudaMemsetAsync(h->d_trace + kChainMaxPhases, 0, col, s) ||
        cudaMemsetAsync(h->d_trace + 2 * kChainMaxPhases, 0xff, col, s) ||
        cudaMemsetAsync(h->d_trace + 3 * kChainMaxPhases, 0,
                        (kChainTraceCols - 3) * col + kEvWords * sizeof(unsigned long long), s))
      return DFLASH_ERR_CUDA;
    P.trace = h->d_trace;
    h->trace_phases = P.pre + 1 + kLayerPhases * c.n_layers + (A.B > 1 && A.ids ? 3 : 0);
  }
  // no LM-head phases when the caller takes the residual only (B = 1, or no ids)
  P.n_phases = P.pre + 1 + kLayerPhases * c.n_layers + (A.B > 1 && A.ids ? 3 : 0);
  P.n_items_max = P.grid + A.batch * c.n_kv_heads;
  P.eps = c.rms_eps;
  P.embed_scale = c.embed_scale;
  P.scale_log2 = 1.4426950408889634f / sqrtf((float)CH_DH);
  P.causal_layers = c.causal_layers, P.window_layers = c.window_layers, P.window = c.sliding_window;
  if (P.grid <= 0) return DFLASH_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.grid);
  cfg.blockDim = dim3(CH_THREADS);
  cfg.dynamicSmemBytes = CH_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  Timer t;
  launch_begin(h, DFLASH_K_DRAFT_CHAIN, s, &t);
  cudaLaunchKernelEx(&cfg, P.pre ? chain_kernel<true> : chain_kernel<false>, P);
  return launch_end(h, s, &t);
}

}  // namespace dflash
