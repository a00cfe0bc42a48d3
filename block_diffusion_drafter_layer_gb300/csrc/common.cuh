// Internal declarations shared by the libdflash translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <vector>

#include "../../include/dflash.h"

namespace dflash {

using bf16 = __nv_bfloat16;

// ---- device status word bits (OR-ed by kernels, read by dflash_get_status)
enum : int {
  ST_CAPACITY = 1,   // a cache append would pass kv->cap
  ST_BOUNDS = 2,     // a token id or position out of range
  ST_TIMEOUT = 4,    // a bounded device wait gave up
};

// ---- conversions ----------------------------------------------------------
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// ---- deterministic block reductions (fixed shuffle tree, then warp 0) ------
// The id an argmax writes.  A row whose logits hold no maximum (all NaN or
// all -inf: only an overflow upstream makes them) leaves the merge's
// sentinel index; the row then gets id 0 (all tied: the lowest index) and
// gap 0, and the status word records ST_BOUNDS instead of an id past the
// vocabulary reaching the caller.
__device__ __forceinline__ int argmax_id(int i1, float& gap, int* status) {
  if (i1 >= 0 && i1 != 0x7fffffff) return i1;
  gap = 0.f;
  atomicOr(status, ST_BOUNDS);
  return 0;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// All threads of the block must call; returns the total to every thread.
__device__ __forceinline__ float block_sum(float v, float* red /* >= 33 floats */) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  if (wid == 0) {
    float t = 0.f;
    for (int i = 0; i < nw; ++i) t += red[i];   // fixed order
    if (lane == 0) red[32] = t;
  }
  __syncthreads();
  return red[32];
}
__device__ __forceinline__ float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  if (wid == 0) {
    float t = -INFINITY;
    for (int i = 0; i < nw; ++i) t = fmaxf(t, red[i]);
    if (lane == 0) red[32] = t;
  }
  __syncthreads();
  return red[32];
}

// ---- which sequence / block position a row belongs to ---------------------
// Uniform: row r is position r % rps of sequence r / rps.
// Ranged:  rows row0[b] .. row0[b]+nrows[b]-1 belong to sequence b.
// A chunk of rows starting at absolute row `offset` maps row r to r + offset.
struct RowMap {
  int ranged;
  int rps;
  const int32_t* row0;
  const int32_t* nrows;
  int batch;
  int offset;
  __device__ __forceinline__ bool map(int r, int& b, int& i) const {
    r += offset;
    if (!ranged) { b = r / rps; i = r - b * rps; return true; }
    for (int s = 0; s < batch; ++s) {
      const int r0 = row0[s], n = nrows[s];
      if (r >= r0 && r < r0 + n) { b = s; i = r - r0; return true; }
    }
    return false;
  }
};

// ---- handle ---------------------------------------------------------------
struct Timer {
  int kclass;
  cudaEvent_t a, b;
};

}  // namespace dflash

namespace dflash {
// TMA descriptors of one layer's bf16 weights (box 64 x 128 rows; SwiGLU
// halves use 64 x 64 so a 128-row tile holds 64 gate + 64 up rows).
struct LayerMaps {
  CUtensorMap wq, wk, wv, wo, wg, wu, wd;
  // boxes for the tensor-core (tcgen05) projection: 64 x 256 rows, and
  // 64 x 128 rows for the SwiGLU gate / up halves
  CUtensorMap tq, tk, tv, to, tg, tu, td;
};
constexpr int kMaxTiles = 8192;   // 128-row weight tiles per projection launch
// d_counters: [0, kMaxTiles) tile arrival counters (tensor-core LM head),
// then the persistent kernel's grid barrier (kMaxTiles + 1) and the
// streaming kernel's grid barrier (kMaxTiles + 2)
// words: per-tile arrival counters; kMaxTiles + 1: the persistent draft
// kernel's grid barrier; + 2: the streaming kernel's; + 3: a word nothing
// writes (the bounded-wait self-test waits on it)
constexpr int kCounters = kMaxTiles + 4;
// phases of the persistent draft-block kernel: 5 of a round, embed, 10 per
// layer, the LM head, its reduce and the merge of its top-2 records
constexpr int kChainMaxPhases = 9 + 10 * DFLASH_MAX_LAYERS;
// timeline columns per phase: first start, last start, first end, last end,
// last CTA done with its multiply-adds, then up to three phase-specific
// marks, each the latest over the grid (projections: first unit done, half
// of the units done; attention: first K/V sub-chunk in, arithmetic done,
// partial written; combine: weights and outputs in)
constexpr int kChainTraceCols = 8;
// per-CTA event log of the persistent kernel (compiled in with
// -DDFLASH_CH_EVLOG=1): kEvCtas sampled CTAs x kChainMaxPhases phases x
// kEvSlots times (ns): 0 start, 1 end, 2.. unit k ready, .. unit k done,
// .. weight load k issued, .. activation load k issued (k < kEvUnits)
constexpr int kEvCtas = 4, kEvUnits = 12, kEvSlots = 2 + 4 * kEvUnits;
constexpr size_t kEvWords = (size_t)kEvCtas * kChainMaxPhases * kEvSlots;
}  // namespace dflash

struct dflash_handle {
  dflash_config cfg;
  dflash_weights w;
  int device = 0;
  int num_sms = 0;
  int* d_status = nullptr;
  int* d_counters = nullptr;       // [kCounters] arrival counters, zero between launches
  float2* d_rope = nullptr;        // [max_pos, d/2] (cos, sin)
  bool have_maps = false;
  bool have_tc = false;
  bool have_wc_map = false;        // d_wmaps holds W_c after the LM head (the round's fusion)
  dflash::LayerMaps maps[DFLASH_MAX_LAYERS];
  CUtensorMap map_wc, map_lm, map_tc_wc, map_tc_lm;
  CUtensorMap* d_wmaps = nullptr;  // device copy: q k v o gate up down per layer, then LM head
  unsigned long long* d_trace = nullptr;  // phase timeline of the persistent kernel, when enabled
  int trace_phases = 0;
  bool timing = false;
  std::vector<cudaEvent_t> free_events;
  std::vector<dflash::Timer> pending;
  double ms[DFLASH_K_NCLASS] = {0};
  int64_t launches[DFLASH_K_NCLASS] = {0};
};

namespace dflash {

// Launch bookkeeping: count, optional event timing, error check.
void launch_begin(dflash_handle* h, int kclass, cudaStream_t s, Timer* t);
int launch_end(dflash_handle* h, cudaStream_t s, Timer* t);
void count_launch();

// Workspace carving (256-byte aligned bump allocator over the caller's buffer).
struct Carve {
  char* base;
  size_t cap, off = 0;
  bool ok = true;
  template <typename T> T* take(size_t n) {
    off = (off + 255) & ~size_t(255);
    T* p = reinterpret_cast<T*>(base + off);
    off += n * sizeof(T);
    if (off > cap) ok = false;
    return p;
  }
};

// ---- weight-streaming projection (k_wstream.cu) ----------------------------
constexpr int WS_MAXMAP = 10;   // weight tensor maps per launch
constexpr int WS_MAXSRC = 5;    // activation sources along K (fused context)
enum SegKind : int { SK_F32 = 0, SK_RESID = 1, SK_HEAD = 2, SK_SWIGLU = 3, SK_ARGMAX = 4 };

// One output segment: tiles [t0, t1) of the launch read weight map `map`
// (and `map2`, the up projection, for SwiGLU) and finish with `kind`.
struct WSeg {
  int t0, t1;
  int kind;
  int map, map2;
  int n_valid;          // valid output columns (features) of the segment
  int d;                // SK_HEAD: head dim
  int rope;             // SK_HEAD: rotate
  const float* gain;    // SK_HEAD: per-head RMSNorm gain, or null
  void* dst;            // output base
  int64_t ld;           // dense output row stride (elements)
  int cache_cap;        // SK_HEAD: > 0 appends into a [batch, heads, cap, d] cache
  int cache_heads;
  int cache_batch;
};

struct WLaunch {
  int nseg = 0;
  WSeg seg[WS_MAXMAP];
  int nmap = 0;
  const CUtensorMap* wmaps[WS_MAXMAP];
  int nsrc = 0;
  const void* a_src[WS_MAXSRC];
  int64_t a_ld = 0;     // activation row stride (elements)
  int K = 0, M = 0;
  RowMap rm{};
  const int32_t* len = nullptr;
  int32_t* ids = nullptr;
  float* gap = nullptr;
  int rps_out = 0;
  const int32_t* anchor = nullptr;
  int bn = 256;         // tcgen05 kernel: output tile width (segment tiles and weight boxes match it)
  bool pair = false;    // tcgen05 kernel: 256-row tiles on CTA pairs (bn 256, weight boxes of 128 rows)
};

// 2-D TMA descriptor with the 128-byte swizzle (box_inner x element size must
// be 128 bytes or less); dtype DFLASH_BF16 or DFLASH_F32.
// swizzle128: 128-byte swizzled boxes (box_inner * element size <= 128);
// false: plain row-major boxes (any inner size up to 256 elements)
bool make_tmap_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                  int dtype = DFLASH_BF16, bool swizzle128 = true);
size_t wstream_scratch_bytes(const dflash_handle* h, int M);
int wstream(dflash_handle* h, cudaStream_t s, int kclass, const WLaunch& L, float* partial,
            float4* amx);

// ---- tensor-core (tcgen05 / TMEM) dense projection (k_tcgemm.cu) ----------
// Same launch description as wstream; 128 x 256 output tiles, SK_F32 and
// SK_HEAD (d = 128) epilogues; segments are in units of 256 columns.
int tc_gemm(dflash_handle* h, cudaStream_t s, int kclass, const WLaunch& L, float4* amx = nullptr);
// CTA pairs of the tcgen05 kernel that can be resident at once (0: none)
int tc_pair_units(const dflash_handle* h);

// ---- split-K attention of the draft block (k_attention.cu) ------------------
size_t attn_scratch_bytes(const dflash_handle* h, int batch, int B);
// Cut the batch's keys into attention items (reads the lengths on the device);
// run once per draft block before the layers' attention_fast calls.
int attn_plan(dflash_handle* h, cudaStream_t s, const int32_t* len, int cap, int batch, int B,
              float* scratch);
bool attn_fast_ok(const dflash_handle* h, int B);
int attention_fast(dflash_handle* h, cudaStream_t s, const void* q, const void* kc, const void* vc,
                   int cap, int kv_batch, const int32_t* len, const void* kb, const void* vb,
                   int batch, int B, void* o, float* scratch, int causal, int window);

// ---- persistent draft block for at most 16 rows (k_chain.cu) ----------------
struct ChainArgs {
  const int32_t* anchor;
  int batch, B;
  const dflash_kv* kv;
  int32_t* ids;
  float* gap;
  float* x;                     // [R, D] fp32 residual
  float* xg;                    // [R, D] fp32 residual x the next RMSNorm's gain
  void *q, *kb, *vb, *o, *a;    // bf16 [R, H*d], [R, G*d] x 2, [R, H*d], [R, F]
  float* ssq;                   // [D / 128, 16] sums of squares, 8 floats apart
  float* partial;               // split-K fix-up tiles
  float* apart;                 // attention run partials (chain_apart_bytes)
  float4* amx;                  // LM-head top-2 records
  // a round (n_in > 0): fuse + inject the pending rows before the block
  int n_in = 0;
  const void* const* hidden = nullptr;   // n_pick device pointers [n_in, D]
  const int32_t* row0 = nullptr;         // device [batch]
  const int32_t* nrow = nullptr;         // device [batch]
  void* ht = nullptr;                    // device bf16 [n_in, D]
};
int chain_grid(const dflash_handle* h);
size_t chain_apart_bytes(const dflash_handle* h, int batch);
bool chain_ok(const dflash_handle* h, int batch, int B);
int draft_chain(dflash_handle* h, cudaStream_t s, const ChainArgs& A);

// ---- kernel launchers (one translation unit each) --------------------------
// A operand source: up to DFLASH_MAX_PICK column segments of width seg
// (column k of row m is seg_ptr[k / seg][m * ld + k % seg]).
struct ASrc {
  const void* p[DFLASH_MAX_PICK];
  int nseg;
  int seg;
  int64_t ld;
};

// C[m, n] (+)= sum_k A[m, k] * W[n, k]; fp32 accumulate in k order.
int gemm(dflash_handle* h, cudaStream_t s, int kclass, int dtype, const ASrc& A,
         const void* W, int64_t ldw, float* C, int64_t ldc, int64_t M, int N, int K,
         bool accumulate);

int embed_block(dflash_handle* h, cudaStream_t s, int dtype, const void* E, const int32_t* anchor,
                int mask_id, int batch, int B, int V, int D, float scale, float* x);
int embed_tokens(dflash_handle* h, cudaStream_t s, int dtype, const void* E, const int32_t* tok,
                 int rows, int V, int D, float scale, float* x);
// out[r] = rmsnorm(in[r]) * g, in fp32 or dtype; rows selected by `skip_every`
// (if > 0, input row r' = r + r / (skip_every - 1) + 1 skips every block's first row).
int rmsnorm_rows(dflash_handle* h, cudaStream_t s, int in_dtype, int out_dtype, const void* in,
                 int64_t ld_in, void* out, int64_t ld_out, const float* g, int64_t rows, int D,
                 float eps, int skip_first_of);
// Per-head (optional RMSNorm) + RoPE on fp32 input [rows, heads*d] -> dtype dst.
int head_norm_rope(dflash_handle* h, cudaStream_t s, int dtype, const float* in, int64_t rows,
                   int heads, int d, const float* gain, bool rope, const RowMap& rm,
                   const int32_t* len, void* dense, void* cache, int cap, int cache_batch);
int swiglu(dflash_handle* h, cudaStream_t s, int dtype, const float* g, const float* u, void* a,
           int64_t n);
int cast_rows(dflash_handle* h, cudaStream_t s, int dtype, const float* in, void* out, int64_t n);
// One bounded wait that nothing completes (see dflash_selftest_wait).
int selftest_wait(dflash_handle* h, cudaStream_t s, int which, int64_t limit_ns);
int advance_len(dflash_handle* h, cudaStream_t s, int32_t* len, const int32_t* nrows, int uniform,
                int batch, int cap);
// Attention of block rows over [cache(0..len) ; block] (draft) or cache(0..pos) (causal target).
int attention(dflash_handle* h, cudaStream_t s, int dtype, const void* q, const void* kc,
              const void* vc, int cap, const int32_t* len, const void* kb, const void* vb,
              int batch, int rows_per_seq, int H, int G, int d, bool causal_in_cache, void* o,
              int causal = 0, int window = 0);
int argmax_rows(dflash_handle* h, cudaStream_t s, const float* logits, int64_t rows, int V,
                int32_t* ids, float* gap, int rows_per_seq_out, const int32_t* anchor);
int verify_greedy(cudaStream_t s, const int32_t* draft, const int32_t* post, int batch, int B,
                  const int32_t* start, int32_t* accept, int32_t* tau, int32_t* bonus,
                  int32_t* out_tokens, int32_t* new_len);
int emit_tokens(cudaStream_t s, const int32_t* out_tokens, const int32_t* tau, int batch, int B,
                int32_t* out_buf, int out_cap, int32_t* out_len, int32_t* tau_log, int log_cap,
                int32_t* n_rounds, int* status);

// ---- sampling at T > 0 (k_sampling.cu) ------------------------------------
size_t sampling_ws_bytes(int rows, int V);
int sample_rows(dflash_handle* h, cudaStream_t s, const float* logits, int rows, int V, float T,
                const double* u, int32_t* ids, int ids_skip_first_of, float* probs, void* ws);
int verify_rejection(dflash_handle* h, cudaStream_t s, const int32_t* draft, const float* q,
                     const float* p, int V, const double* u_acc, const double* u_smp, int batch,
                     int B, const int32_t* start, int32_t* accept, int32_t* tau, int32_t* token,
                     int32_t* out_tokens, int32_t* new_len, void* ws);
int conv_corr(dflash_handle* h, cudaStream_t s, const float* x, const void* kp, int64_t R,
              float* corr);
int conv_apply(dflash_handle* h, cudaStream_t s, const float* y, const float* corr,
               const float* base, int call, int64_t R, int B, float* out, bool accumulate);
size_t select_ws_bytes(int batch, int B, int V, int D, int K, int rank);
bool select_shape_ok(int B, int V, int D, int K, int rank);
int select_candidates(dflash_handle* h, cudaStream_t s, const float* logits, const float* x,
                      const float* gain, const int32_t* anchor, int batch, int B, int K,
                      const void* w_h, int rank, const void* code_pred, const void* code_succ,
                      int n_codes, int32_t* draft_ids, int32_t* cand_out, float* scores,
                      void* ws);

}  // namespace dflash
