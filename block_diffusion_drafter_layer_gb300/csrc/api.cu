// C ABI of libdflash: argument validation, workspace layout and the order of
// kernels for each call of the DFlash draft path.
#include <atomic>
#include <cmath>
#include <cstring>
#include <vector>

#include <cudaTypedefs.h>

#include "common.cuh"

namespace dflash {

static std::atomic<int64_t> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static cudaEvent_t take_event(dflash_handle* h) {
  if (!h->free_events.empty()) {
    cudaEvent_t e = h->free_events.back();
    h->free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

void launch_begin(dflash_handle* h, int kclass, cudaStream_t s, Timer* t) {
  t->kclass = kclass;
  t->a = t->b = nullptr;
  if (h && h->timing) {
    t->a = take_event(h);
    cudaEventRecord(t->a, s);
  }
}

int launch_end(dflash_handle* h, cudaStream_t s, Timer* t) {
  count_launch();
  const cudaError_t e = cudaGetLastError();
  if (h && t->a) {
    t->b = take_event(h);
    cudaEventRecord(t->b, s);
    h->pending.push_back(*t);
  }
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

// A draft layer's mask (txtmix §6): causal rows, and the window of keys
// (0: none).
static int layer_causal(const dflash_config& c, int l) { return (c.causal_layers >> l) & 1; }
static int layer_window(const dflash_config& c, int l) {
  return ((c.window_layers >> l) & 1) ? c.sliding_window : 0;
}

static size_t esize(int dtype) { return dtype == DFLASH_BF16 ? 2 : 4; }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Rows of fuse / inject processed per pass (bounds the fp32 staging buffers).
constexpr int64_t kChunkRows = 4096;

static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Scratch of the weight-streaming kernel: two fp32 partial tiles per CTA and
// one top-2 record per (vocabulary tile, row).
static size_t ws_partial_bytes(const dflash_handle* h) {
  return round256(wstream_scratch_bytes(h, 64));
}
static size_t ws_amx_bytes(const dflash_handle* h, int64_t R = 64) {
  const size_t a = (size_t)((h->cfg.vocab + 127) / 128) * 64;        // streaming kernel
  const size_t b = (size_t)((h->cfg.vocab + 255) / 256) * std::max<int64_t>(R, 64);  // tcgen05
  const size_t c = (size_t)std::max(chain_grid(h), 2 * h->num_sms) * 16;  // persistent kernel
  return round256(std::max({a, b, c}) * sizeof(float4));
}

// Split-K attention partials of the draft block; the same region holds the
// persistent kernel's attention-run partials.
static size_t attn_region_bytes(const dflash_handle* h, int batch, int B) {
  return round256(std::max(attn_scratch_bytes(h, batch, B), chain_apart_bytes(h, batch)));
}

// Workspace of a forward pass (draft block, target forward, LM head) over R rows.
static size_t forward_bytes(const dflash_config& c, int64_t R) {
  const size_t sz = esize(c.dtype);
  const int64_t D = c.hidden, Hd = (int64_t)c.n_heads * c.head_dim,
                Gd = (int64_t)c.n_kv_heads * c.head_dim, F = c.ffn, V = c.vocab;
  size_t b = 0;
  b += round256(R * F * sz);          // a (SwiGLU output)
  b += round256(R * D * 4) * 2;       // x, x times the next norm gain
  b += round256(R * std::max(D, F) * sz);  // h / a
  b += round256(R * Hd * 4);          // qf
  b += round256(R * Gd * 4) * 2;      // kf, vf
  b += round256(R * Hd * sz);         // q
  b += round256(R * Gd * sz) * 2;     // kb, vb
  b += round256(R * Hd * sz);         // o
  b += round256(R * F * 4) * 2;       // gf, uf
  b += round256(R * D * sz);          // hf
  b += round256(R * V * 4);           // logits
  if (c.conv_group > 0) {             // conv: prepared rows / sublayer outputs, corrections
    b += round256(R * D * 4);
    b += round256(R * (4 * D / c.conv_group) * 4);
  }
  return b + 1024;
}

// Per-row workspace of fuse / inject passes.
static size_t chunk_row_bytes(const dflash_config& c) {
  const int64_t D = c.hidden, Gd = (int64_t)c.n_kv_heads * c.head_dim;
  return (size_t)std::max<int64_t>(D * 4, 2 * Gd * 4);
}

struct Fwd {
  float *x, *xg, *qf, *kf, *vf, *gf, *uf, *logits, *partial, *attn, *ssq;
  float *cu, *cc;   // conv: prepared rows / sublayer outputs [R, D], corrections [R, 4 D / group]
  float4* amx;
  void *h, *q, *kb, *vb, *o, *hf, *a;
};

static bool carve_forward(const dflash_handle* h, int64_t R, void* ws, size_t ws_bytes, Fwd* f,
                          int batch = 0, int B = 0) {
  const dflash_config& c = h->cfg;
  const size_t sz = esize(c.dtype);
  const int64_t D = c.hidden, Hd = (int64_t)c.n_heads * c.head_dim,
                Gd = (int64_t)c.n_kv_heads * c.head_dim, F = c.ffn, V = c.vocab;
  Carve cv{(char*)ws, ws_bytes};
  f->partial = cv.take<float>(ws_partial_bytes(h) / sizeof(float));
  f->attn = batch > 0 ? cv.take<float>(attn_region_bytes(h, batch, B) / sizeof(float)) : nullptr;
  f->ssq = cv.take<float>((size_t)(h->cfg.hidden / 128 + 1) * 16 * 8);
  f->amx = cv.take<float4>(ws_amx_bytes(h, R) / sizeof(float4));
  f->a = cv.take<char>(R * F * sz);
  f->x = cv.take<float>(R * D);
  f->xg = cv.take<float>(R * D);
  f->h = cv.take<char>(R * std::max(D, F) * sz);
  f->qf = cv.take<float>(R * Hd);
  f->kf = cv.take<float>(R * Gd);
  f->vf = cv.take<float>(R * Gd);
  f->q = cv.take<char>(R * Hd * sz);
  f->kb = cv.take<char>(R * Gd * sz);
  f->vb = cv.take<char>(R * Gd * sz);
  f->o = cv.take<char>(R * Hd * sz);
  f->gf = cv.take<float>(R * F);
  f->uf = cv.take<float>(R * F);
  f->hf = cv.take<char>(R * D * sz);
  f->logits = cv.take<float>(R * V);
  f->cu = f->cc = nullptr;
  if (c.conv_group > 0) {
    f->cu = cv.take<float>(R * D);
    f->cc = cv.take<float>(R * (4 * D / c.conv_group));
  }
  return cv.ok;
}

static ASrc one_src(const void* p, int64_t ld, int K) {
  ASrc a{};
  a.p[0] = p;
  a.nseg = 1;
  a.seg = K;
  a.ld = ld;
  return a;
}

static const char* byte_off(const void* p, int64_t elems, int dtype) {
  return (const char*)p + elems * (int64_t)esize(dtype);
}

// SwiGLU FFN + o_proj residual of one layer (shared by draft and target).
static int mlp_tail(dflash_handle* h, cudaStream_t s, const dflash_layer_weights& L, Fwd& f,
                    int64_t R) {
  const dflash_config& c = h->cfg;
  const int D = c.hidden, F = c.ffn, Hd = c.n_heads * c.head_dim, dt = c.dtype;
  int rc;
  if ((rc = gemm(h, s, DFLASH_K_WEIGHT_GEMM, dt, one_src(f.o, Hd, Hd), L.wo, Hd, f.x, D, R, D, Hd,
                 true)))
    return rc;
  if ((rc = rmsnorm_rows(h, s, DFLASH_F32, dt, f.x, D, f.h, D, L.g_post, R, D, c.rms_eps, 0)))
    return rc;
  if ((rc = gemm(h, s, DFLASH_K_WEIGHT_GEMM, dt, one_src(f.h, D, D), L.wg, D, f.gf, F, R, F, D,
                 false)))
    return rc;
  if ((rc = gemm(h, s, DFLASH_K_WEIGHT_GEMM, dt, one_src(f.h, D, D), L.wu, D, f.uf, F, R, F, D,
                 false)))
    return rc;
  if ((rc = swiglu(h, s, dt, f.gf, f.uf, f.h, R * F))) return rc;
  return gemm(h, s, DFLASH_K_WEIGHT_GEMM, dt, one_src(f.h, F, F), L.wd, F, f.x, D, R, D, F, true);
}

// mlp_tail with the conv modules (txtmix §13-§14): x += finish(o W_o^T);
// then h = norm(prepare(x)) with the FFN module's corrections and
// x += finish(SwiGLU FFN of h).  Each finish call convolves the sublayer
// output across adjacent rows of a block, so it follows the projection
// instead of being its epilogue.
static int conv_mlp_tail(dflash_handle* h, cudaStream_t s, const dflash_layer_weights& L, Fwd& f,
                         int64_t R, int B) {
  const dflash_config& c = h->cfg;
  const int D = c.hidden, F = c.ffn, Hd = c.n_heads * c.head_dim, dt = c.dtype;
  int rc;
  if ((rc = gemm(h, s, DFLASH_K_WEIGHT_GEMM, dt, one_src(f.o, Hd, Hd), L.wo, Hd, f.cu, D, R, D, Hd,
                 false)))
    return rc;
  if ((rc = conv_apply(h, s, f.cu, f.cc, L.conv_att_base, 1, R, B, f.x, true))) return rc;
  if ((rc = conv_corr(h, s, f.x, L.conv_mlp_kp, R, f.cc))) return rc;
  if ((rc = conv_apply(h, s, f.x, f.cc, L.conv_mlp_base, 0, R, B, f.cu, false))) return rc;
  if ((rc = rmsnorm_rows(h, s, DFLASH_F32, dt, f.cu, D, f.h, D, L.g_post, R, D, c.rms_eps, 0)))
    return rc;
  if ((rc = gemm(h, s, DFLASH_K_WEIGHT_GEMM, dt, one_src(f.h, D, D), L.wg, D, f.gf, F, R, F, D,
                 false)))
    return rc;
  if ((rc = gemm(h, s, DFLASH_K_WEIGHT_GEMM, dt, one_src(f.h, D, D), L.wu, D, f.uf, F, R, F, D,
                 false)))
    return rc;
  if ((rc = swiglu(h, s, dt, f.gf, f.uf, f.h, R * F))) return rc;
  if ((rc = gemm(h, s, DFLASH_K_WEIGHT_GEMM, dt, one_src(f.h, F, F), L.wd, F, f.cu, D, R, D, F,
                 false)))
    return rc;
  return conv_apply(h, s, f.cu, f.cc, L.conv_mlp_base, 1, R, B, f.x, true);
}

static bool streaming(const dflash_handle* h, int64_t M);
static bool dense_tc(const dflash_handle* h, int64_t M);
static int lm_head_tc(dflash_handle* h, cudaStream_t s, Fwd& f, int64_t rows, int32_t* ids,
                      float* gap, int rps_out, const int32_t* anchor);
static int lm_head_stream(dflash_handle* h, cudaStream_t s, Fwd& f, int64_t rows, int32_t* ids,
                          float* gap, int rps_out, const int32_t* anchor);

#ifndef DFLASH_LM_TC_MIN_ROWS
#define DFLASH_LM_TC_MIN_ROWS 33
#endif
static int lm_head(dflash_handle* h, cudaStream_t s, Fwd& f, const float* x, int64_t rows,
                   const float* gain, int skip_first_of, int32_t* ids, float* gap, int rps_out,
                   const int32_t* anchor) {
  const dflash_config& c = h->cfg;
  const int D = c.hidden, V = c.vocab, dt = c.dtype;
  int rc;
  if ((rc = rmsnorm_rows(h, s, DFLASH_F32, dt, x, D, f.hf, D, gain, rows, D, c.rms_eps,
                         skip_first_of)))
    return rc;
  // From DFLASH_LM_TC_MIN_ROWS rows the LM head (a weight of vocabulary x D)
  // goes to the tensor cores: the streaming kernel's warp-level MMAs bound it
  // there, not HBM
  if (h->have_tc && rows >= DFLASH_LM_TC_MIN_ROWS)
    return lm_head_tc(h, s, f, rows, ids, gap, rps_out, anchor);
  if (streaming(h, rows)) return lm_head_stream(h, s, f, rows, ids, gap, rps_out, anchor);
  if (dense_tc(h, rows)) return lm_head_tc(h, s, f, rows, ids, gap, rps_out, anchor);
  if ((rc = gemm(h, s, DFLASH_K_LM_HEAD, dt, one_src(f.hf, D, D), h->w.lm_head, D, f.logits, V,
                 rows, V, D, false)))
    return rc;
  return argmax_rows(h, s, f.logits, rows, V, ids, gap, rps_out, anchor);
}

// ---- weight-streaming paths (bf16, at most 64 activation rows) -------------
// Row counts (compile-time tuning): the weight-streaming kernel takes
// projections of at most DFLASH_STREAM_MAX_ROWS rows, the tensor-core kernel
// those of at least DFLASH_TC_MIN_ROWS rows (when both apply, streaming).
#ifndef DFLASH_STREAM_MAX_ROWS
#define DFLASH_STREAM_MAX_ROWS 64
#endif
#ifndef DFLASH_TC_MIN_ROWS
#define DFLASH_TC_MIN_ROWS 128
#endif
static bool streaming(const dflash_handle* h, int64_t M) {
  return h->have_maps && M >= 1 && M <= DFLASH_STREAM_MAX_ROWS;
}

static WSeg make_seg(int t0, int t1, int kind, int map, int n_valid, void* dst, int64_t ld) {
  WSeg g{};
  g.t0 = t0;
  g.t1 = t1;
  g.kind = kind;
  g.map = map;
  g.n_valid = n_valid;
  g.dst = dst;
  g.ld = ld;
  return g;
}

static WSeg head_seg(int t0, int t1, int map, int n_valid, int d, int rope, const float* gain,
                     void* dst, int64_t ld) {
  WSeg g = make_seg(t0, t1, SK_HEAD, map, n_valid, dst, ld);
  g.d = d;
  g.rope = rope;
  g.gain = gain;
  return g;
}

// q, k, v of the block rows in one launch; the epilogue applies the per-head
// q/k RMSNorm and RoPE and stores bf16 heads for the attention kernel.
static int qkv_stream(dflash_handle* h, cudaStream_t s, int l, Fwd& f, int64_t R, const RowMap& rm,
                      const int32_t* len) {
  const dflash_config& c = h->cfg;
  const dflash_layer_weights& W = h->w.layers[l];
  const int D = c.hidden, d = c.head_dim, Hd = c.n_heads * d, Gd = c.n_kv_heads * d;
  const int tq = Hd / 128, tk = Gd / 128;
  WLaunch L;
  L.nmap = 3;
  L.wmaps[0] = &h->maps[l].wq;
  L.wmaps[1] = &h->maps[l].wk;
  L.wmaps[2] = &h->maps[l].wv;
  L.nseg = 3;
  L.seg[0] = head_seg(0, tq, 0, Hd, d, 1, c.qk_norm ? W.q_norm : nullptr, f.q, Hd);
  L.seg[1] = head_seg(tq, tq + tk, 1, Gd, d, 1, c.qk_norm ? W.k_norm : nullptr, f.kb, Gd);
  L.seg[2] = head_seg(tq + tk, tq + 2 * tk, 2, Gd, d, 0, nullptr, f.vb, Gd);
  L.nsrc = 1;
  L.a_src[0] = f.h;
  L.a_ld = D;
  L.K = D;
  L.M = (int)R;
  L.rm = rm;
  L.len = len;
  return wstream(h, s, DFLASH_K_WEIGHT_GEMM, L, f.partial, f.amx);
}

// o_proj (+ residual), RMSNorm, gate/up with the SwiGLU epilogue, down (+ residual).
// With the conv modules (conv): o_proj and down store plain rows into f.cu
// and their finish convs add them into x; the FFN's norm reads the rows of
// its prepare conv.
static int mlp_stream(dflash_handle* h, cudaStream_t s, int l, Fwd& f, int64_t R, bool conv,
                      int B) {
  const dflash_config& c = h->cfg;
  const dflash_layer_weights& W = h->w.layers[l];
  const int D = c.hidden, F = c.ffn, Hd = c.n_heads * c.head_dim, dt = c.dtype;
  int rc;
  WLaunch L;
  L.nmap = 1;
  L.wmaps[0] = &h->maps[l].wo;
  L.nseg = 1;
  L.seg[0] = conv ? make_seg(0, (D + 127) / 128, SK_F32, 0, D, f.cu, D)
                  : make_seg(0, (D + 127) / 128, SK_RESID, 0, D, f.x, D);
  L.nsrc = 1;
  L.a_src[0] = f.o;
  L.a_ld = Hd;
  L.K = Hd;
  L.M = (int)R;
  if ((rc = wstream(h, s, DFLASH_K_WEIGHT_GEMM, L, f.partial, f.amx))) return rc;
  if (conv) {
    if ((rc = conv_apply(h, s, f.cu, f.cc, W.conv_att_base, 1, R, B, f.x, true))) return rc;
    if ((rc = conv_corr(h, s, f.x, W.conv_mlp_kp, R, f.cc))) return rc;
    if ((rc = conv_apply(h, s, f.x, f.cc, W.conv_mlp_base, 0, R, B, f.cu, false))) return rc;
  }
  if ((rc = rmsnorm_rows(h, s, DFLASH_F32, dt, conv ? f.cu : f.x, D, f.h, D, W.g_post, R, D,
                         c.rms_eps, 0)))
    return rc;
  WLaunch G;
  G.nmap = 2;
  G.wmaps[0] = &h->maps[l].wg;
  G.wmaps[1] = &h->maps[l].wu;
  G.nseg = 1;
  G.seg[0] = make_seg(0, (F + 63) / 64, SK_SWIGLU, 0, F, f.a, F);
  G.seg[0].map2 = 1;
  G.nsrc = 1;
  G.a_src[0] = f.h;
  G.a_ld = D;
  G.K = D;
  G.M = (int)R;
  if ((rc = wstream(h, s, DFLASH_K_WEIGHT_GEMM, G, f.partial, f.amx))) return rc;
  WLaunch Dn;
  Dn.nmap = 1;
  Dn.wmaps[0] = &h->maps[l].wd;
  Dn.nseg = 1;
  Dn.seg[0] = conv ? make_seg(0, (D + 127) / 128, SK_F32, 0, D, f.cu, D)
                   : make_seg(0, (D + 127) / 128, SK_RESID, 0, D, f.x, D);
  Dn.nsrc = 1;
  Dn.a_src[0] = f.a;
  Dn.a_ld = F;
  Dn.K = F;
  Dn.M = (int)R;
  if ((rc = wstream(h, s, DFLASH_K_WEIGHT_GEMM, Dn, f.partial, f.amx))) return rc;
  return conv ? conv_apply(h, s, f.cu, f.cc, W.conv_mlp_base, 1, R, B, f.x, true) : DFLASH_OK;
}

static int lm_head_stream(dflash_handle* h, cudaStream_t s, Fwd& f, int64_t rows, int32_t* ids,
                          float* gap, int rps_out, const int32_t* anchor) {
  const dflash_config& c = h->cfg;
  WLaunch L;
  L.nmap = 1;
  L.wmaps[0] = &h->map_lm;
  L.nseg = 1;
  L.seg[0] = make_seg(0, (c.vocab + 127) / 128, SK_ARGMAX, 0, c.vocab, nullptr, 0);
  L.nsrc = 1;
  L.a_src[0] = f.hf;
  L.a_ld = c.hidden;
  L.K = c.hidden;
  L.M = (int)rows;
  L.ids = ids;
  L.gap = gap;
  L.rps_out = rps_out;
  L.anchor = anchor;
  return wstream(h, s, DFLASH_K_LM_HEAD, L, f.partial, f.amx);
}

// ---- tensor-core paths for blocks of >= 128 rows (e.g. batch 32 x B 16) -----
// Output tile width of a tcgen05 projection with N output columns: 128 where
// 128-column tiles still fit in one wave (256-column tiles would leave more
// than half of the SMs idle: o_proj and down at batch 32 x B 16), else 256.
static int tc_width(const dflash_handle* h, int64_t M, int64_t N) {
  return 2 * ((M + 127) / 128) * (N / 256) <= h->num_sms ? 128 : 256;
}

static int qkv_tc(dflash_handle* h, cudaStream_t s, int l, Fwd& f, int64_t R, const RowMap& rm,
                  const int32_t* len) {
  const dflash_config& c = h->cfg;
  const dflash_layer_weights& W = h->w.layers[l];
  const int D = c.hidden, d = c.head_dim, Hd = c.n_heads * d, Gd = c.n_kv_heads * d;
  WLaunch L;
  L.bn = tc_width(h, R, Hd + 2 * Gd);
  const int tq = Hd / L.bn, tk = Gd / L.bn;
  const bool narrow = L.bn == 128;
  L.nmap = 3;
  L.wmaps[0] = narrow ? &h->maps[l].wq : &h->maps[l].tq;
  L.wmaps[1] = narrow ? &h->maps[l].wk : &h->maps[l].tk;
  L.wmaps[2] = narrow ? &h->maps[l].wv : &h->maps[l].tv;
  L.nseg = 3;
  L.seg[0] = head_seg(0, tq, 0, Hd, d, 1, c.qk_norm ? W.q_norm : nullptr, f.q, Hd);
  L.seg[1] = head_seg(tq, tq + tk, 1, Gd, d, 1, c.qk_norm ? W.k_norm : nullptr, f.kb, Gd);
  L.seg[2] = head_seg(tq + tk, tq + 2 * tk, 2, Gd, d, 0, nullptr, f.vb, Gd);
  L.nsrc = 1;
  L.a_src[0] = f.h;
  L.a_ld = D;
  L.K = D;
  L.M = (int)R;
  L.rm = rm;
  L.len = len;
  return tc_gemm(h, s, DFLASH_K_WEIGHT_GEMM, L);
}

static int mlp_tc(dflash_handle* h, cudaStream_t s, int l, Fwd& f, int64_t R) {
  const dflash_config& c = h->cfg;
  const dflash_layer_weights& W = h->w.layers[l];
  const int D = c.hidden, F = c.ffn, Hd = c.n_heads * c.head_dim, dt = c.dtype;
  int rc;
  WLaunch L;
  L.bn = tc_width(h, R, D);
  L.nmap = 1;
  L.wmaps[0] = L.bn == 128 ? &h->maps[l].wo : &h->maps[l].to;
  L.nseg = 1;
  L.seg[0] = make_seg(0, D / L.bn, SK_RESID, 0, D, f.x, D);
  L.nsrc = 1;
  L.a_src[0] = f.o;
  L.a_ld = Hd;
  L.K = Hd;
  L.M = (int)R;
  if ((rc = tc_gemm(h, s, DFLASH_K_WEIGHT_GEMM, L))) return rc;
  if ((rc = rmsnorm_rows(h, s, DFLASH_F32, dt, f.x, D, f.h, D, W.g_post, R, D, c.rms_eps, 0)))
    return rc;
  WLaunch G;
  G.bn = tc_width(h, R, 2 * (int64_t)F);
  G.nmap = 2;
  G.wmaps[0] = G.bn == 128 ? &h->maps[l].wg : &h->maps[l].tg;   // gate / up boxes of bn / 2 rows
  G.wmaps[1] = G.bn == 128 ? &h->maps[l].wu : &h->maps[l].tu;
  G.nseg = 1;
  G.seg[0] = make_seg(0, F / (G.bn / 2), SK_SWIGLU, 0, F, f.a, F);
  G.seg[0].map2 = 1;
  G.nsrc = 1;
  G.a_src[0] = f.h;
  G.a_ld = D;
  G.K = D;
  G.M = (int)R;
  if ((rc = tc_gemm(h, s, DFLASH_K_WEIGHT_GEMM, G))) return rc;
  WLaunch Dn;
  Dn.bn = tc_width(h, R, D);
  Dn.nmap = 1;
  Dn.wmaps[0] = Dn.bn == 128 ? &h->maps[l].wd : &h->maps[l].td;
  Dn.nseg = 1;
  Dn.seg[0] = make_seg(0, D / Dn.bn, SK_RESID, 0, D, f.x, D);
  Dn.nsrc = 1;
  Dn.a_src[0] = f.a;
  Dn.a_ld = F;
  Dn.K = F;
  Dn.M = (int)R;
  return tc_gemm(h, s, DFLASH_K_WEIGHT_GEMM, Dn);
}

static int lm_head_tc(dflash_handle* h, cudaStream_t s, Fwd& f, int64_t rows, int32_t* ids,
                      float* gap, int rps_out, const int32_t* anchor) {
  const dflash_config& c = h->cfg;
  WLaunch L;
  L.nmap = 1;
  L.wmaps[0] = &h->map_tc_lm;
  L.nseg = 1;
  L.seg[0] = make_seg(0, (c.vocab + 255) / 256, SK_ARGMAX, 0, c.vocab, nullptr, 0);
  L.nsrc = 1;
  L.a_src[0] = f.hf;
  L.a_ld = c.hidden;
  L.K = c.hidden;
  L.M = (int)rows;
  L.ids = ids;
  L.gap = gap;
  L.rps_out = rps_out;
  L.anchor = anchor;
  return tc_gemm(h, s, DFLASH_K_LM_HEAD, L, f.amx);
}

// fp32 logits of rows through the final RMSNorm (gain) and the shared LM
// head: the same projections as lm_head with the fp32-store epilogue.
static int lm_logits(dflash_handle* h, cudaStream_t s, Fwd& f, const float* x, int64_t rows,
                     const float* gain, int skip_first_of, float* logits) {
  const dflash_config& c = h->cfg;
  const int D = c.hidden, V = c.vocab, dt = c.dtype;
  int rc;
  if ((rc = rmsnorm_rows(h, s, DFLASH_F32, dt, x, D, f.hf, D, gain, rows, D, c.rms_eps,
                         skip_first_of)))
    return rc;
  if (streaming(h, rows) && V % 4 == 0) {
    WLaunch L;
    L.nmap = 1;
    L.wmaps[0] = &h->map_lm;
    L.nseg = 1;
    L.seg[0] = make_seg(0, (V + 127) / 128, SK_F32, 0, V, logits, V);
    L.nsrc = 1;
    L.a_src[0] = f.hf;
    L.a_ld = D;
    L.K = D;
    L.M = (int)rows;
    return wstream(h, s, DFLASH_K_LM_HEAD, L, f.partial, nullptr);
  }
  if (dense_tc(h, rows) && V % 32 == 0) {
    WLaunch L;
    L.nmap = 1;
    L.wmaps[0] = &h->map_tc_lm;
    L.nseg = 1;
    L.seg[0] = make_seg(0, (V + 255) / 256, SK_F32, 0, V, logits, V);
    L.nsrc = 1;
    L.a_src[0] = f.hf;
    L.a_ld = D;
    L.K = D;
    L.M = (int)rows;
    return tc_gemm(h, s, DFLASH_K_LM_HEAD, L);
  }
  return gemm(h, s, DFLASH_K_LM_HEAD, dt, one_src(f.hf, D, D), h->w.lm_head, D, logits, V, rows,
              V, D, false);
}

static bool kv_ok(const dflash_handle* h, const dflash_kv* kv, int batch) {
  if (!kv || !kv->len || kv->cap <= 0 || kv->batch_cap < batch) return false;
  for (int l = 0; l < h->cfg.n_layers; ++l)
    if (!kv->k[l] || !kv->v[l] || !aligned16(kv->k[l]) || !aligned16(kv->v[l])) return false;
  return true;
}

// TMA descriptors of every bf16 weight, built once per handle.  Shapes that
// do not tile into 128-row / 64-column blocks keep the portable kernels.
static bool make_weight_maps(dflash_handle* h) {
  const dflash_config& c = h->cfg;
  const dflash_weights& w = h->w;
  const int64_t D = c.hidden, d = c.head_dim, Hd = c.n_heads * d, Gd = c.n_kv_heads * d,
                F = c.ffn, V = c.vocab;
  if (c.dtype != DFLASH_BF16 || D % 128 || Hd % 128 || Gd % 128 || F % 64 || h->num_sms < 1)
    return false;
  auto mk = [](CUtensorMap* m, const void* p, int64_t rows, int64_t cols, uint32_t box_rows) {
    return make_tmap_2d(m, p, (uint64_t)cols, (uint64_t)rows, (uint64_t)cols * 2, 64, box_rows);
  };
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash_layer_weights& L = w.layers[l];
    LayerMaps& M = h->maps[l];
    if (!mk(&M.wq, L.wq, Hd, D, 128) || !mk(&M.wk, L.wk, Gd, D, 128) ||
        !mk(&M.wv, L.wv, Gd, D, 128) || !mk(&M.wo, L.wo, D, Hd, 128) ||
        !mk(&M.wg, L.wg, F, D, 64) || !mk(&M.wu, L.wu, F, D, 64) || !mk(&M.wd, L.wd, D, F, 128))
      return false;
  }
  if (w.wc && !mk(&h->map_wc, w.wc, D, c.n_pick * D, 128)) return false;
  if (!mk(&h->map_lm, w.lm_head, V, D, 128)) return false;
  h->have_maps = true;
  // device copy of the draft-layer and LM-head maps for the persistent kernel
  if (d == 128 && F % 64 == 0) {
    std::vector<CUtensorMap> tab((size_t)c.n_layers * 7 + 2);
    for (int l = 0; l < c.n_layers; ++l) {
      const LayerMaps& M = h->maps[l];
      const CUtensorMap* src[7] = {&M.wq, &M.wk, &M.wv, &M.wo, &M.wg, &M.wu, &M.wd};
      for (int k = 0; k < 7; ++k) tab[(size_t)l * 7 + k] = *src[k];
    }
    tab[(size_t)c.n_layers * 7] = h->map_lm;
    tab[(size_t)c.n_layers * 7 + 1] = w.wc ? h->map_wc : h->map_lm;
    void* p = nullptr;
    if (cudaMalloc(&p, tab.size() * sizeof(CUtensorMap)) == cudaSuccess) {
      if (cudaMemcpy(p, tab.data(), tab.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice) ==
          cudaSuccess) {
        h->d_wmaps = (CUtensorMap*)p;
        h->have_wc_map = w.wc != nullptr && c.hidden % 128 == 0;
      } else {
        cudaFree(p);
      }
    }
  }
  // 256-row boxes for the tensor-core projection of long prefixes
  if (d == 128 && D % 256 == 0 && Hd % 256 == 0 && Gd % 256 == 0 && F % 128 == 0) {
    bool ok = mk(&h->map_tc_lm, w.lm_head, V, D, 256);
    if (ok && w.wc) ok = mk(&h->map_tc_wc, w.wc, D, c.n_pick * D, 256);
    for (int l = 0; ok && l < c.n_layers; ++l) {
      const dflash_layer_weights& L = w.layers[l];
      LayerMaps& M = h->maps[l];
      ok = mk(&M.tq, L.wq, Hd, D, 256) && mk(&M.tk, L.wk, Gd, D, 256) &&
           mk(&M.tv, L.wv, Gd, D, 256) && mk(&M.to, L.wo, D, Hd, 256) &&
           mk(&M.tg, L.wg, F, D, 128) && mk(&M.tu, L.wu, F, D, 128) &&
           mk(&M.td, L.wd, D, F, 256);
    }
    h->have_tc = ok;
  }
  return true;
}

// Long prefixes (>= 128 rows) of a bf16 handle go to the tensor-core kernel.
static bool dense_tc(const dflash_handle* h, int64_t M) {
  return h->have_tc && M >= DFLASH_TC_MIN_ROWS;
}

}  // namespace dflash

using namespace dflash;

extern "C" {

const char* dflash_strerror(int code) {
  switch (code) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_INVALID_ARG: return "invalid argument";
    case DFLASH_ERR_SHAPE: return "unsupported shape";
    case DFLASH_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case DFLASH_ERR_CAPACITY: return "K/V cache capacity exceeded";
    case DFLASH_ERR_UNSUPPORTED: return "unsupported dtype, head_dim or device";
    case DFLASH_ERR_CUDA: return "CUDA error";
    case DFLASH_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case DFLASH_ERR_DEVICE_BOUNDS: return "token id or position out of range";
    case DFLASH_ERR_WORKSPACE: return "workspace too small";
    case DFLASH_ERR_STATIC_LIMIT: return "request exceeds the fixed internal scratch limits";
    default: return "unknown error";
  }
}

int64_t dflash_launch_count(void) { return g_launches.load(); }

int dflash_build_target_layer_ids(int32_t n_target_layers, int32_t n_pick, int32_t* ids_out) {
  if (!ids_out || n_pick < 1 || n_pick > DFLASH_MAX_PICK) return DFLASH_ERR_INVALID_ARG;
  if (n_pick == 1) {
    ids_out[0] = n_target_layers / 2;
    return DFLASH_OK;
  }
  const int lo = 1, hi = n_target_layers - 3;
  if (hi < lo) return DFLASH_ERR_SHAPE;
  const int64_t span = hi - lo;
  for (int i = 0; i < n_pick; ++i)
    ids_out[i] = lo + (int32_t)((2 * i * span + (n_pick - 1)) / (2 * (n_pick - 1)));
  return DFLASH_OK;
}

int dflash_create(const dflash_config* cfg, const dflash_weights* w, dflash_handle** out) {
  if (!cfg || !w || !out) return DFLASH_ERR_INVALID_ARG;
  *out = nullptr;
  const dflash_config& c = *cfg;
  if (c.dtype != DFLASH_F32 && c.dtype != DFLASH_BF16) return DFLASH_ERR_UNSUPPORTED;
  if (c.head_dim != 64 && c.head_dim != 128) return DFLASH_ERR_UNSUPPORTED;
  if (c.hidden <= 0 || c.hidden % 8 || c.n_heads <= 0 || c.n_kv_heads <= 0 ||
      c.n_heads % c.n_kv_heads || c.ffn <= 0 || c.ffn % 8 || c.vocab <= 0 || c.n_layers < 1 ||
      c.n_layers > DFLASH_MAX_LAYERS || c.n_pick < 1 || c.n_pick > DFLASH_MAX_PICK ||
      c.max_pos <= 0 || c.mask_token_id < 0 || c.mask_token_id >= c.vocab || !(c.rms_eps > 0.f))
    return DFLASH_ERR_SHAPE;
  if (!w->embed || !w->lm_head || !w->g_f) return DFLASH_ERR_INVALID_ARG;
  if (c.causal_layers < 0 || c.window_layers < 0 || c.sliding_window < 0 ||
      (c.window_layers != 0 && c.sliding_window < 1) ||
      ((c.causal_layers | c.window_layers) >> c.n_layers) != 0 || c.conv_group < 0 ||
      (c.conv_group > 0 && c.hidden % c.conv_group != 0))
    return DFLASH_ERR_SHAPE;
  const void* al[] = {w->embed, w->lm_head, w->wc};
  for (const void* p : al)
    if (p && !aligned16(p)) return DFLASH_ERR_ALIGNMENT;
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash_layer_weights& L = w->layers[l];
    const void* ps[] = {L.wq, L.wk, L.wv, L.wo, L.wg, L.wu, L.wd};
    for (const void* p : ps) {
      if (!p) return DFLASH_ERR_INVALID_ARG;
      if (!aligned16(p)) return DFLASH_ERR_ALIGNMENT;
    }
    if (!L.g_in || !L.g_post) return DFLASH_ERR_INVALID_ARG;
    if (c.qk_norm && (!L.q_norm || !L.k_norm)) return DFLASH_ERR_INVALID_ARG;
    if (c.conv_group > 0 &&
        (!L.conv_att_kp || !L.conv_att_base || !L.conv_mlp_kp || !L.conv_mlp_base))
      return DFLASH_ERR_INVALID_ARG;
  }
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DFLASH_ERR_CUDA;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return DFLASH_ERR_UNSUPPORTED;

  dflash_handle* h = new dflash_handle();
  h->cfg = c;
  h->w = *w;
  h->device = dev;
  cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaMalloc(&h->d_status, sizeof(int)) != cudaSuccess ||
      cudaMalloc(&h->d_counters, kCounters * sizeof(int)) != cudaSuccess) {
    cudaFree(h->d_status);
    delete h;
    return DFLASH_ERR_CUDA;
  }
  cudaMemset(h->d_status, 0, sizeof(int));
  cudaMemset(h->d_counters, 0, kCounters * sizeof(int));
  if (!make_weight_maps(h)) h->have_maps = false;
  // RoPE table: angle pos * theta^(-2i/d) in double precision, stored as fp32.
  const int half = c.head_dim / 2;
  std::vector<float2> tab((size_t)c.max_pos * half);
  for (int64_t p = 0; p < c.max_pos; ++p)
    for (int i = 0; i < half; ++i) {
      const double ang =
          (double)p * std::pow((double)c.rope_theta, -2.0 * (double)i / (double)c.head_dim);
      tab[(size_t)p * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
    }
  if (cudaMalloc(&h->d_rope, tab.size() * sizeof(float2)) != cudaSuccess ||
      cudaMemcpy(h->d_rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) !=
          cudaSuccess) {
    cudaFree(h->d_status);
    cudaFree(h->d_counters);
    cudaFree(h->d_rope);
    delete h;
    return DFLASH_ERR_CUDA;
  }
  *out = h;
  return DFLASH_OK;
}

int dflash_destroy(dflash_handle* h) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  for (auto& t : h->pending) {
    cudaEventDestroy(t.a);
    cudaEventDestroy(t.b);
  }
  for (auto e : h->free_events) cudaEventDestroy(e);
  cudaFree(h->d_status);
  cudaFree(h->d_counters);
  cudaFree(h->d_rope);
  cudaFree(h->d_wmaps);
  cudaFree(h->d_trace);
  delete h;
  return DFLASH_OK;
}

size_t dflash_workspace_bytes(const dflash_handle* h, int32_t max_batch, int32_t max_block,
                              int64_t max_rows) {
  if (!h || max_batch < 0 || max_block < 0 || max_rows < 0) return 0;
  const int64_t R = std::max<int64_t>({(int64_t)max_batch * max_block, max_rows, 1});
  // a forward pass over R rows, or fuse / inject in full kChunkRows passes
  const size_t scratch = ws_partial_bytes(h) + ws_amx_bytes(h, R) + 1024 +
                         round256((size_t)(h->cfg.hidden / 128 + 1) * 16 * 8 * sizeof(float)) +
                         (max_batch > 0 && max_block > 0
                              ? attn_region_bytes(h, max_batch, max_block) : 0);
  const size_t fwd = forward_bytes(h->cfg, R);
  const size_t chunk = round256(kChunkRows * chunk_row_bytes(h->cfg)) + 1024;
  return std::max(fwd, chunk) + scratch;
}

int dflash_fuse_context(dflash_handle* h, const void* const* hidden, int64_t T, void* h_t_out,
                        void* ws, size_t ws_bytes, dflash_stream_t st) {
  if (!h || !hidden || T < 0) return DFLASH_ERR_INVALID_ARG;
  if (!h->w.wc || !h->w.g_c) return DFLASH_ERR_INVALID_ARG;
  if (T == 0) return DFLASH_OK;
  if (!h_t_out || !ws) return DFLASH_ERR_INVALID_ARG;
  const dflash_config& c = h->cfg;
  for (int i = 0; i < c.n_pick; ++i) {
    if (!hidden[i]) return DFLASH_ERR_INVALID_ARG;
    if (!aligned16(hidden[i])) return DFLASH_ERR_ALIGNMENT;
  }
  if (!aligned16(h_t_out) || !aligned16(ws)) return DFLASH_ERR_ALIGNMENT;
  cudaStream_t s = (cudaStream_t)st;
  const int D = c.hidden, dt = c.dtype;
  if (streaming(h, T)) {
    Carve cv{(char*)ws, ws_bytes};
    float* partial = cv.take<float>(ws_partial_bytes(h) / sizeof(float));
    float* Y = cv.take<float>(T * D);
    if (!cv.ok) return DFLASH_ERR_WORKSPACE;
    WLaunch L;
    L.nmap = 1;
    L.wmaps[0] = &h->map_wc;
    L.nseg = 1;
    L.seg[0] = make_seg(0, (D + 127) / 128, SK_F32, 0, D, Y, D);
    L.nsrc = c.n_pick;
    for (int i = 0; i < c.n_pick; ++i) L.a_src[i] = hidden[i];
    L.a_ld = D;
    L.K = c.n_pick * D;
    L.M = (int)T;
    int rc = wstream(h, s, DFLASH_K_DENSE_GEMM, L, partial, nullptr);
    if (rc) return rc;
    return rmsnorm_rows(h, s, DFLASH_F32, dt, Y, D, h_t_out, D, h->w.g_c, T, D, c.rms_eps, 0);
  }
  if (dense_tc(h, T)) {
    // tensor-core projection in row chunks staged as fp32 in the workspace,
    // each followed by the row RMSNorm
    const int64_t fit = (int64_t)(ws_bytes / ((size_t)D * 4 + 1)) / 128 * 128;
    const int64_t chunk = std::min<int64_t>(T, fit);
    if (fit < std::min<int64_t>(T, 128)) return DFLASH_ERR_WORKSPACE;
    float* Yc = (float*)ws;
    for (int64_t r0 = 0; r0 < T; r0 += chunk) {
      const int64_t n = std::min(chunk, T - r0);
      WLaunch L;
      L.nmap = 1;
      // CTA pairs load half of a 256-column tile's weight rows each
      L.pair = tc_pair_units(h) > 0;
      L.wmaps[0] = L.pair ? &h->map_wc : &h->map_tc_wc;
      L.nseg = 1;
      L.seg[0] = make_seg(0, D / 256, SK_F32, 0, D, Yc, D);
      L.nsrc = c.n_pick;
      for (int i = 0; i < c.n_pick; ++i) L.a_src[i] = byte_off(hidden[i], r0 * D, dt);
      L.a_ld = D;
      L.K = c.n_pick * D;
      L.M = (int)n;
      int rc = tc_gemm(h, s, DFLASH_K_DENSE_GEMM, L);
      if (rc) return rc;
      rc = rmsnorm_rows(h, s, DFLASH_F32, dt, Yc, D, (void*)byte_off(h_t_out, r0 * D, dt), D,
                        h->w.g_c, n, D, c.rms_eps, 0);
      if (rc) return rc;
    }
    return DFLASH_OK;
  }
  const int64_t chunk = std::min<int64_t>(kChunkRows, (int64_t)(ws_bytes / (D * 4 + 1)));
  if (chunk < 1) return DFLASH_ERR_WORKSPACE;
  float* Y = (float*)ws;
  for (int64_t r0 = 0; r0 < T; r0 += chunk) {
    const int64_t n = std::min(chunk, T - r0);
    ASrc a{};
    for (int i = 0; i < c.n_pick; ++i) a.p[i] = byte_off(hidden[i], r0 * D, dt);
    a.nseg = c.n_pick;
    a.seg = D;
    a.ld = D;
    int rc = gemm(h, s, DFLASH_K_DENSE_GEMM, dt, a, h->w.wc, (int64_t)c.n_pick * D, Y, D, n, D,
                  c.n_pick * D, false);
    if (rc) return rc;
    rc = rmsnorm_rows(h, s, DFLASH_F32, dt, Y, D, (void*)byte_off(h_t_out, r0 * D, dt), D, h->w.g_c,
                      n, D, c.rms_eps, 0);
    if (rc) return rc;
  }
  return DFLASH_OK;
}

int dflash_inject_kv(dflash_handle* h, const void* h_t, int64_t n_rows, const int32_t* seq_row0,
                     const int32_t* seq_rows, int32_t batch, const dflash_kv* kv, void* ws,
                     size_t ws_bytes, dflash_stream_t st) {
  if (!h || !h_t || !seq_row0 || !seq_rows || !ws || n_rows < 0 || batch < 1)
    return DFLASH_ERR_INVALID_ARG;
  if (!kv_ok(h, kv, batch)) return DFLASH_ERR_INVALID_ARG;
  if (!aligned16(h_t) || !aligned16(ws)) return DFLASH_ERR_ALIGNMENT;
  cudaStream_t s = (cudaStream_t)st;
  const dflash_config& c = h->cfg;
  const int D = c.hidden, G = c.n_kv_heads, d = c.head_dim, Gd = G * d, dt = c.dtype;
  if (n_rows == 0) return advance_len(h, s, kv->len, seq_rows, 0, batch, kv->cap);
  if (streaming(h, n_rows)) {
    Carve cv{(char*)ws, ws_bytes};
    float* partial = cv.take<float>(ws_partial_bytes(h) / sizeof(float));
    if (!cv.ok) return DFLASH_ERR_WORKSPACE;
    const int tk = Gd / 128;
    const RowMap rm{1, 0, seq_row0, seq_rows, batch, 0};
    for (int l0 = 0; l0 < c.n_layers; l0 += WS_MAXMAP / 2) {
      const int nl = std::min(WS_MAXMAP / 2, c.n_layers - l0);
      WLaunch L;
      L.nmap = 2 * nl;
      L.nseg = 2 * nl;
      for (int j = 0; j < nl; ++j) {
        const int l = l0 + j;
        L.wmaps[2 * j] = &h->maps[l].wk;
        L.wmaps[2 * j + 1] = &h->maps[l].wv;
        WSeg gk = head_seg(2 * j * tk, (2 * j + 1) * tk, 2 * j, Gd, d, 1,
                           c.qk_norm ? h->w.layers[l].k_norm : nullptr, kv->k[l], 0);
        WSeg gv = head_seg((2 * j + 1) * tk, (2 * j + 2) * tk, 2 * j + 1, Gd, d, 0, nullptr,
                           kv->v[l], 0);
        gk.cache_cap = gv.cache_cap = kv->cap;
        gk.cache_heads = gv.cache_heads = G;
        gk.cache_batch = gv.cache_batch = kv->batch_cap;
        L.seg[2 * j] = gk;
        L.seg[2 * j + 1] = gv;
      }
      L.nsrc = 1;
      L.a_src[0] = h_t;
      L.a_ld = D;
      L.K = D;
      L.M = (int)n_rows;
      L.rm = rm;
      L.len = kv->len;
      const int rc = wstream(h, s, DFLASH_K_DENSE_GEMM, L, partial, nullptr);
      if (rc) return rc;
    }
    return advance_len(h, s, kv->len, seq_rows, 0, batch, kv->cap);
  }
  if (dense_tc(h, n_rows) && n_rows <= 0x7fffffff) {
    // one tensor-core launch for every layer's k and v; the epilogue applies
    // k_norm and RoPE and appends to the caches
    const int tk = Gd / 256;
    const RowMap rm{1, 0, seq_row0, seq_rows, batch, 0};
    for (int l0 = 0; l0 < c.n_layers; l0 += WS_MAXMAP / 2) {
      const int nl = std::min(WS_MAXMAP / 2, c.n_layers - l0);
      WLaunch L;
      L.nmap = 2 * nl;
      L.nseg = 2 * nl;
      for (int j = 0; j < nl; ++j) {
        const int l = l0 + j;
        L.wmaps[2 * j] = &h->maps[l].tk;
        L.wmaps[2 * j + 1] = &h->maps[l].tv;
        WSeg gk = head_seg(2 * j * tk, (2 * j + 1) * tk, 2 * j, Gd, d, 1,
                           c.qk_norm ? h->w.layers[l].k_norm : nullptr, kv->k[l], 0);
        WSeg gv = head_seg((2 * j + 1) * tk, (2 * j + 2) * tk, 2 * j + 1, Gd, d, 0, nullptr,
                           kv->v[l], 0);
        gk.cache_cap = gv.cache_cap = kv->cap;
        gk.cache_heads = gv.cache_heads = G;
        gk.cache_batch = gv.cache_batch = kv->batch_cap;
        L.seg[2 * j] = gk;
        L.seg[2 * j + 1] = gv;
      }
      L.nsrc = 1;
      L.a_src[0] = h_t;
      L.a_ld = D;
      L.K = D;
      L.M = (int)n_rows;
      L.rm = rm;
      L.len = kv->len;
      const int rc = tc_gemm(h, s, DFLASH_K_DENSE_GEMM, L);
      if (rc) return rc;
    }
    return advance_len(h, s, kv->len, seq_rows, 0, batch, kv->cap);
  }
  const int64_t chunk = std::min<int64_t>(kChunkRows, (int64_t)(ws_bytes / (2 * Gd * 4 + 512)));
  if (chunk < 1) return DFLASH_ERR_WORKSPACE;
  Carve cv{(char*)ws, ws_bytes};
  float* kf = cv.take<float>(chunk * Gd);
  float* vf = cv.take<float>(chunk * Gd);
  if (!cv.ok) return DFLASH_ERR_WORKSPACE;
  for (int64_t r0 = 0; r0 < n_rows; r0 += chunk) {
    const int64_t n = std::min(chunk, n_rows - r0);
    RowMap rm{1, 0, seq_row0, seq_rows, batch, (int)r0};
    const ASrc a = one_src(byte_off(h_t, r0 * D, dt), D, D);
    for (int l = 0; l < c.n_layers; ++l) {
      const dflash_layer_weights& L = h->w.layers[l];
      int rc;
      if ((rc = gemm(h, s, DFLASH_K_DENSE_GEMM, dt, a, L.wk, D, kf, Gd, n, Gd, D, false))) return rc;
      if ((rc = gemm(h, s, DFLASH_K_DENSE_GEMM, dt, a, L.wv, D, vf, Gd, n, Gd, D, false))) return rc;
      if ((rc = head_norm_rope(h, s, dt, kf, n, G, d, c.qk_norm ? L.k_norm : nullptr, true, rm,
                               kv->len, nullptr, kv->k[l], kv->cap, kv->batch_cap)))
        return rc;
      if ((rc = head_norm_rope(h, s, dt, vf, n, G, d, nullptr, false, rm, kv->len, nullptr,
                               kv->v[l], kv->cap, kv->batch_cap)))
        return rc;
    }
  }
  return advance_len(h, s, kv->len, seq_rows, 0, batch, kv->cap);
}

int dflash_draft_block(dflash_handle* h, const int32_t* anchor, int32_t batch, int32_t B,
                       const dflash_kv* kv, int32_t* draft_ids, float* top2_gap, float* hidden_out,
                       void* ws, size_t ws_bytes, dflash_stream_t st) {
  if (!h || !anchor || (!draft_ids && !hidden_out) || !ws || batch < 1 || B < 1)
    return DFLASH_ERR_INVALID_ARG;
  if (!kv_ok(h, kv, batch)) return DFLASH_ERR_INVALID_ARG;
  if (!aligned16(ws)) return DFLASH_ERR_ALIGNMENT;
  cudaStream_t s = (cudaStream_t)st;
  const dflash_config& c = h->cfg;
  const int D = c.hidden, H = c.n_heads, G = c.n_kv_heads, d = c.head_dim, dt = c.dtype;
  const int Hd = H * d, Gd = G * d;
  const int64_t R = (int64_t)batch * B;
  Fwd f;
  if (!carve_forward(h, R, ws, ws_bytes, &f, batch, B)) return DFLASH_ERR_WORKSPACE;
  int rc;
  if (chain_ok(h, batch, B)) {
    // the whole block in one persistent launch
    ChainArgs A{anchor, batch, B, kv, draft_ids, top2_gap, f.x, f.xg, f.q, f.kb, f.vb, f.o, f.a,
                f.ssq, f.partial, f.attn, f.amx};
    if ((rc = draft_chain(h, s, A))) return rc;
    if (hidden_out &&
        cudaMemcpyAsync(hidden_out, f.x, R * D * sizeof(float), cudaMemcpyDeviceToDevice, s))
      return DFLASH_ERR_CUDA;
    if (B == 1 && draft_ids &&
        cudaMemcpyAsync(draft_ids, anchor, batch * sizeof(int32_t), cudaMemcpyDeviceToDevice, s))
      return DFLASH_ERR_CUDA;
    return DFLASH_OK;
  }
  if ((rc = embed_block(h, s, dt, h->w.embed, anchor, c.mask_token_id, batch, B, c.vocab, D,
                        c.embed_scale, f.x)))
    return rc;
  const RowMap rm{0, B, nullptr, nullptr, batch, 0};
  const bool conv = c.conv_group > 0;   // conv modules: streaming or SIMT projections
  const bool stream = streaming(h, R);
  const bool tcore = !conv && !stream && dense_tc(h, R) && attn_fast_ok(h, B);
  if ((tcore || stream) && attn_fast_ok(h, B) &&
      (rc = attn_plan(h, s, kv->len, kv->cap, batch, B, f.attn)))
    return rc;
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash_layer_weights& L = h->w.layers[l];
    if (conv) {   // the attention module's corrections and prepare call: h = norm(prepare(x))
      if ((rc = conv_corr(h, s, f.x, L.conv_att_kp, R, f.cc))) return rc;
      if ((rc = conv_apply(h, s, f.x, f.cc, L.conv_att_base, 0, R, B, f.cu, false))) return rc;
    }
    if ((rc = rmsnorm_rows(h, s, DFLASH_F32, dt, conv ? f.cu : f.x, D, f.h, D, L.g_in, R, D,
                           c.rms_eps, 0)))
      return rc;
    if (tcore) {
      if ((rc = qkv_tc(h, s, l, f, R, rm, kv->len))) return rc;
      if ((rc = attention_fast(h, s, f.q, kv->k[l], kv->v[l], kv->cap, kv->batch_cap, kv->len, f.kb, f.vb, batch,
                               B, f.o, f.attn, layer_causal(c, l), layer_window(c, l))))
        return rc;
      if ((rc = mlp_tc(h, s, l, f, R))) return rc;
      continue;
    }
    if (stream) {
      if ((rc = qkv_stream(h, s, l, f, R, rm, kv->len))) return rc;
      if (attn_fast_ok(h, B))
        rc = attention_fast(h, s, f.q, kv->k[l], kv->v[l], kv->cap, kv->batch_cap, kv->len, f.kb, f.vb, batch, B,
                            f.o, f.attn, layer_causal(c, l), layer_window(c, l));
      else
        rc = attention(h, s, dt, f.q, kv->k[l], kv->v[l], kv->cap, kv->len, f.kb, f.vb, batch, B,
                       H, G, d, false, f.o, layer_causal(c, l), layer_window(c, l));
      if (rc) return rc;
      if ((rc = mlp_stream(h, s, l, f, R, conv, B))) return rc;
      continue;
    }
    const ASrc a = one_src(f.h, D, D);
    if ((rc = gemm(h, s, DFLASH_K_WEIGHT_GEMM, dt, a, L.wq, D, f.qf, Hd, R, Hd, D, false))) return rc;
    if ((rc = gemm(h, s, DFLASH_K_WEIGHT_GEMM, dt, a, L.wk, D, f.kf, Gd, R, Gd, D, false))) return rc;
    if ((rc = gemm(h, s, DFLASH_K_WEIGHT_GEMM, dt, a, L.wv, D, f.vf, Gd, R, Gd, D, false))) return rc;
    if ((rc = head_norm_rope(h, s, dt, f.qf, R, H, d, c.qk_norm ? L.q_norm : nullptr, true, rm,
                             kv->len, f.q, nullptr, 0, 0)))
      return rc;
    if ((rc = head_norm_rope(h, s, dt, f.kf, R, G, d, c.qk_norm ? L.k_norm : nullptr, true, rm,
                             kv->len, f.kb, nullptr, 0, 0)))
      return rc;
    if ((rc = head_norm_rope(h, s, dt, f.vf, R, G, d, nullptr, false, rm, kv->len, f.vb, nullptr, 0,
                             0)))
      return rc;
    if ((rc = attention(h, s, dt, f.q, kv->k[l], kv->v[l], kv->cap, kv->len, f.kb, f.vb, batch, B,
                        H, G, d, false, f.o, layer_causal(c, l), layer_window(c, l))))
      return rc;
    if ((rc = conv ? conv_mlp_tail(h, s, L, f, R, B) : mlp_tail(h, s, L, f, R))) return rc;
  }
  if (hidden_out &&
      cudaMemcpyAsync(hidden_out, f.x, R * D * sizeof(float), cudaMemcpyDeviceToDevice, s))
    return DFLASH_ERR_CUDA;
  if (!draft_ids) return DFLASH_OK;   // the residual only (the caller samples)
  if (B == 1) {
    if (cudaMemcpyAsync(draft_ids, anchor, batch * sizeof(int32_t), cudaMemcpyDeviceToDevice, s))
      return DFLASH_ERR_CUDA;
    return DFLASH_OK;
  }
  return lm_head(h, s, f, f.x, (int64_t)batch * (B - 1), h->w.g_f, B, draft_ids, top2_gap, B,
                 anchor);
}

int dflash_draft_round(dflash_handle* h, const void* const* hidden, int32_t n_rows,
                       const int32_t* seq_row0, const int32_t* seq_rows, void* h_t_out,
                       const int32_t* anchor, int32_t batch, int32_t B, const dflash_kv* kv,
                       int32_t* draft_ids, float* top2_gap, float* hidden_out, void* ws,
                       size_t ws_bytes, dflash_stream_t st) {
  if (!h || n_rows < 0) return DFLASH_ERR_INVALID_ARG;
  if (n_rows == 0)
    return dflash_draft_block(h, anchor, batch, B, kv, draft_ids, top2_gap, hidden_out, ws,
                              ws_bytes, st);
  if (!hidden || !seq_row0 || !seq_rows || !h_t_out || !anchor || (!draft_ids && !hidden_out) ||
      !ws || batch < 1 || B < 1)
    return DFLASH_ERR_INVALID_ARG;
  if (!kv_ok(h, kv, batch)) return DFLASH_ERR_INVALID_ARG;
  const dflash_config& c = h->cfg;
  for (int i = 0; i < c.n_pick; ++i) {
    if (!hidden[i]) return DFLASH_ERR_INVALID_ARG;
    if (!aligned16(hidden[i])) return DFLASH_ERR_ALIGNMENT;
  }
  if (!aligned16(h_t_out) || !aligned16(ws)) return DFLASH_ERR_ALIGNMENT;
  cudaStream_t s = (cudaStream_t)st;
  if (chain_ok(h, batch, B) && n_rows <= 16 && h->have_wc_map && h->w.g_c &&
      aligned16(h->w.g_c)) {
    // fusion, injection and the block in one persistent launch
    const int64_t R = (int64_t)batch * B;
    Fwd f;
    if (!carve_forward(h, std::max<int64_t>(R, n_rows), ws, ws_bytes, &f, batch, B))
      return DFLASH_ERR_WORKSPACE;
    ChainArgs A{anchor, batch, B, kv, draft_ids, top2_gap, f.x, f.xg, f.q, f.kb, f.vb, f.o, f.a,
                f.ssq, f.partial, f.attn, f.amx};
    A.n_in = n_rows;
    A.hidden = hidden;
    A.row0 = seq_row0;
    A.nrow = seq_rows;
    A.ht = h_t_out;
    int rc = draft_chain(h, s, A);
    if (rc) return rc;
    if (hidden_out &&
        cudaMemcpyAsync(hidden_out, f.x, R * c.hidden * sizeof(float), cudaMemcpyDeviceToDevice, s))
      return DFLASH_ERR_CUDA;
    if (B == 1 && draft_ids &&
        cudaMemcpyAsync(draft_ids, anchor, batch * sizeof(int32_t), cudaMemcpyDeviceToDevice, s))
      return DFLASH_ERR_CUDA;
    return DFLASH_OK;
  }
  int rc = dflash_fuse_context(h, hidden, n_rows, h_t_out, ws, ws_bytes, st);
  if (!rc) rc = dflash_inject_kv(h, h_t_out, n_rows, seq_row0, seq_rows, batch, kv, ws, ws_bytes, st);
  if (!rc)
    rc = dflash_draft_block(h, anchor, batch, B, kv, draft_ids, top2_gap, hidden_out, ws, ws_bytes,
                            st);
  return rc;
}

int dflash_verify_greedy(const int32_t* draft, const int32_t* post, int32_t batch, int32_t B,
                         const int32_t* start, int32_t* accept, int32_t* tau, int32_t* bonus,
                         int32_t* out_tokens, int32_t* new_len, dflash_stream_t st) {
  if (!draft || !post || !start || !accept || !bonus || !out_tokens || batch < 0 || B < 1)
    return DFLASH_ERR_INVALID_ARG;
  if (batch == 0) return DFLASH_OK;
  return verify_greedy((cudaStream_t)st, draft, post, batch, B, start, accept, tau, bonus,
                       out_tokens, new_len);
}

int dflash_emit_tokens(dflash_handle* h, const int32_t* out_tokens, const int32_t* tau,
                       int32_t batch, int32_t B, int32_t* out_buf, int32_t out_cap,
                       int32_t* out_len, int32_t* tau_log, int32_t log_cap, int32_t* n_rounds,
                       dflash_stream_t st) {
  if (!h || !out_tokens || !tau || !out_buf || !out_len || batch < 1 || B < 1 || out_cap < 1 ||
      (tau_log && (!n_rounds || log_cap < 1)))
    return DFLASH_ERR_INVALID_ARG;
  return emit_tokens((cudaStream_t)st, out_tokens, tau, batch, B, out_buf, out_cap, out_len,
                     tau_log, log_cap, n_rounds, h->d_status);
}

int64_t dflash_round_out_len(int32_t batch, int32_t B) {
  if (batch < 1 || B < 1) return -1;
  const int64_t P = ((int64_t)batch + 3) / 4 * 4;
  return 2 * (int64_t)batch * B + 3 * P;
}

int dflash_round_host(dflash_handle* h, const void* host_features, void* dev_features,
                      int32_t n_rows, const int32_t* host_in, int32_t* dev_in, int32_t* host_out,
                      int32_t* dev_out, const int32_t* seq_row0, const int32_t* seq_rows,
                      void* h_t_out, int32_t batch, int32_t B, const dflash_kv* kv,
                      const int32_t* start, int32_t* new_len, void* ws, size_t ws_bytes,
                      dflash_stream_t st) {
  if (!h || n_rows < 0 || batch < 1 || B < 1 || !host_in || !dev_in || !host_out || !dev_out ||
      !start || (n_rows > 0 && (!host_features || !dev_features)))
    return DFLASH_ERR_INVALID_ARG;
  const dflash_config& c = h->cfg;
  if (c.n_pick < 1 || c.n_pick > 8) return DFLASH_ERR_INVALID_ARG;
  if ((n_rows > 0 && !aligned16(dev_features)) || !aligned16(dev_out)) return DFLASH_ERR_ALIGNMENT;
  cudaStream_t s = (cudaStream_t)st;
  const int64_t slice = (int64_t)n_rows * c.hidden * esize(c.dtype);
  const int64_t n_in = (int64_t)batch + (int64_t)batch * B;
  const int64_t n_out = dflash_round_out_len(batch, B);
  if (n_rows > 0 && cudaMemcpyAsync(dev_features, host_features, slice * c.n_pick,
                                    cudaMemcpyHostToDevice, s))
    return DFLASH_ERR_CUDA;
  if (cudaMemcpyAsync(dev_in, host_in, n_in * sizeof(int32_t), cudaMemcpyHostToDevice, s))
    return DFLASH_ERR_CUDA;
  const void* hidden[8] = {};
  for (int i = 0; i < c.n_pick && n_rows > 0; ++i)
    hidden[i] = (const char*)dev_features + i * slice;
  const int64_t bB = (int64_t)batch * B, P = ((int64_t)batch + 3) / 4 * 4;
  int32_t* ids = dev_out;
  int32_t* tokens = dev_out + bB;
  int32_t* accept = dev_out + 2 * bB;
  int rc = dflash_draft_round(h, n_rows ? hidden : nullptr, n_rows, seq_row0, seq_rows, h_t_out,
                              dev_in, batch, B, kv, ids, nullptr, nullptr, ws, ws_bytes, st);
  if (rc) return rc;
  rc = dflash_verify_greedy(ids, dev_in + batch, batch, B, start, accept, accept + P, accept + 2 * P,
                            tokens, new_len, st);
  if (rc) return rc;
  if (cudaMemcpyAsync(host_out, dev_out, n_out * sizeof(int32_t), cudaMemcpyDeviceToHost, s))
    return DFLASH_ERR_CUDA;
  return DFLASH_OK;
}

int dflash_lm_head_argmax(dflash_handle* h, const float* x, int32_t rows, const float* norm_gain,
                          int32_t* ids, float* top2_gap, void* ws, size_t ws_bytes,
                          dflash_stream_t st) {
  if (!h || !x || !norm_gain || !ids || !ws || rows < 0) return DFLASH_ERR_INVALID_ARG;
  if (rows == 0) return DFLASH_OK;
  Fwd f;
  if (!carve_forward(h, rows, ws, ws_bytes, &f)) return DFLASH_ERR_WORKSPACE;
  return lm_head(h, (cudaStream_t)st, f, x, rows, norm_gain, 0, ids, top2_gap, 0, nullptr);
}

int dflash_lm_head_logits(dflash_handle* h, const float* x, int32_t rows, const float* norm_gain,
                          int32_t skip_first_of, float* logits, void* ws, size_t ws_bytes,
                          dflash_stream_t st) {
  if (!h || !x || !norm_gain || !logits || !ws || rows < 0 || skip_first_of < 0 ||
      skip_first_of == 1)
    return DFLASH_ERR_INVALID_ARG;
  if (rows == 0) return DFLASH_OK;
  if (!aligned16(logits) || !aligned16(ws)) return DFLASH_ERR_ALIGNMENT;
  Fwd f;
  if (!carve_forward(h, rows, ws, ws_bytes, &f)) return DFLASH_ERR_WORKSPACE;
  return lm_logits(h, (cudaStream_t)st, f, x, rows, norm_gain, skip_first_of, logits);
}

size_t dflash_sampling_ws_bytes(int32_t rows, int32_t vocab) {
  if (rows < 0 || vocab < 1) return 0;
  return sampling_ws_bytes(rows, vocab);
}

int dflash_sample_rows(dflash_handle* h, const float* logits, int32_t rows, int32_t vocab,
                       float temperature, const double* u, int32_t* ids,
                       int32_t ids_skip_first_of, float* probs, void* ws, size_t ws_bytes,
                       dflash_stream_t st) {
  if (!h || !logits || rows < 0 || vocab < 1 || !(temperature > 0.f) || (!ids && !probs) ||
      (ids && !u) || ids_skip_first_of < 0 || ids_skip_first_of == 1 || !ws)
    return DFLASH_ERR_INVALID_ARG;
  if (((uintptr_t)ws & 255) != 0) return DFLASH_ERR_ALIGNMENT;
  if (ws_bytes < sampling_ws_bytes(rows, vocab)) return DFLASH_ERR_WORKSPACE;
  if (rows == 0) return DFLASH_OK;
  return sample_rows(h, (cudaStream_t)st, logits, rows, vocab, temperature, u, ids,
                     ids_skip_first_of, probs, ws);
}

int dflash_verify_rejection(dflash_handle* h, const int32_t* draft, const float* q_probs,
                            const float* p_probs, int32_t vocab, const double* u_accept,
                            const double* u_sample, int32_t batch, int32_t B,
                            const int32_t* start, int32_t* accept, int32_t* tau, int32_t* token,
                            int32_t* out_tokens, int32_t* new_len, void* ws, size_t ws_bytes,
                            dflash_stream_t st) {
  if (!h || !draft || !q_probs || !p_probs || vocab < 1 || !u_sample || batch < 1 || B < 1 ||
      (B > 1 && !u_accept) || !start || !accept || !out_tokens || !ws)
    return DFLASH_ERR_INVALID_ARG;
  if (((uintptr_t)ws & 255) != 0) return DFLASH_ERR_ALIGNMENT;
  if (ws_bytes < sampling_ws_bytes(batch, vocab)) return DFLASH_ERR_WORKSPACE;
  return verify_rejection(h, (cudaStream_t)st, draft, q_probs, p_probs, vocab, u_accept, u_sample,
                          batch, B, start, accept, tau, token, out_tokens, new_len, ws);
}

size_t dflash_select_ws_bytes(const dflash_handle* h, int32_t batch, int32_t B, int32_t top_k,
                              int32_t rank) {
  if (!h || batch < 1 || B < 2 || top_k < 1 || rank < 1) return 0;
  return select_ws_bytes(batch, B, h->cfg.vocab, h->cfg.hidden, top_k, rank);
}

int dflash_select_candidates(dflash_handle* h, const float* logits, const float* hidden,
                             const float* norm_gain, const int32_t* anchor, int32_t batch,
                             int32_t B, int32_t top_k, const void* w_h, int32_t rank,
                             const void* code_pred, const void* code_succ, int32_t n_codes,
                             int32_t* draft_ids, int32_t* candidates, float* scores, void* ws,
                             size_t ws_bytes, dflash_stream_t st) {
  if (!h || !logits || !hidden || !norm_gain || !anchor || !w_h || !code_pred || !code_succ ||
      !draft_ids || !ws || batch < 1 || n_codes < h->cfg.vocab ||
      !select_shape_ok(B, h->cfg.vocab, h->cfg.hidden, top_k, rank))
    return DFLASH_ERR_INVALID_ARG;
  if (((uintptr_t)ws & 255) != 0 || !aligned16(hidden) || !aligned16(norm_gain) ||
      !aligned16(w_h))
    return DFLASH_ERR_ALIGNMENT;
  if (ws_bytes < select_ws_bytes(batch, B, h->cfg.vocab, h->cfg.hidden, top_k, rank))
    return DFLASH_ERR_WORKSPACE;
  return select_candidates(h, (cudaStream_t)st, logits, hidden, norm_gain, anchor, batch, B, top_k,
                           w_h, rank, code_pred, code_succ, n_codes, draft_ids, candidates,
                           scores, ws);
}

int dflash_target_forward(dflash_handle* h, const int32_t* tokens, int32_t batch, int32_t T,
                          const dflash_kv* kv, const int32_t* tap_ids, int32_t n_taps,
                          void* taps_out, int32_t* argmax_out, void* ws, size_t ws_bytes,
                          dflash_stream_t st) {
  if (!h || !tokens || !argmax_out || !ws || batch < 1 || T < 1 || n_taps < 0)
    return DFLASH_ERR_INVALID_ARG;
  if (n_taps > 0 && (!tap_ids || !taps_out)) return DFLASH_ERR_INVALID_ARG;
  if (!kv_ok(h, kv, batch)) return DFLASH_ERR_INVALID_ARG;
  const dflash_config& c = h->cfg;
  for (int j = 0; j < n_taps; ++j)
    if (tap_ids[j] < 0 || tap_ids[j] >= c.n_layers) return DFLASH_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)st;
  const int D = c.hidden, H = c.n_heads, G = c.n_kv_heads, d = c.head_dim, dt = c.dtype;
  const int Hd = H * d, Gd = G * d;
  const int64_t R = (int64_t)batch * T;
  Fwd f;
  if (!carve_forward(h, R, ws, ws_bytes, &f)) return DFLASH_ERR_WORKSPACE;
  int rc;
  if ((rc = embed_tokens(h, s, dt, h->w.embed, tokens, (int)R, c.vocab, D, c.embed_scale, f.x)))
    return rc;
  const RowMap rm{0, T, nullptr, nullptr, batch, 0};
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash_layer_weights& L = h->w.layers[l];
    if ((rc = rmsnorm_rows(h, s, DFLASH_F32, dt, f.x, D, f.h, D, L.g_in, R, D, c.rms_eps, 0)))
      return rc;
    const ASrc a = one_src(f.h, D, D);
    if ((rc = gemm(h, s, DFLASH_K_WEIGHT_GEMM, dt, a, L.wq, D, f.qf, Hd, R, Hd, D, false))) return rc;
    if ((rc = gemm(h, s, DFLASH_K_WEIGHT_GEMM, dt, a, L.wk, D, f.kf, Gd, R, Gd, D, false))) return rc;
    if ((rc = gemm(h, s, DFLASH_K_WEIGHT_GEMM, dt, a, L.wv, D, f.vf, Gd, R, Gd, D, false))) return rc;
    if ((rc = head_norm_rope(h, s, dt, f.qf, R, H, d, c.qk_norm ? L.q_norm : nullptr, true, rm,
                             kv->len, f.q, nullptr, 0, 0)))
      return rc;
    if ((rc = head_norm_rope(h, s, dt, f.kf, R, G, d, c.qk_norm ? L.k_norm : nullptr, true, rm,
                             kv->len, nullptr, kv->k[l], kv->cap, kv->batch_cap)))
      return rc;
    if ((rc = head_norm_rope(h, s, dt, f.vf, R, G, d, nullptr, false, rm, kv->len, nullptr,
                             kv->v[l], kv->cap, kv->batch_cap)))
      return rc;
    if ((rc = attention(h, s, dt, f.q, kv->k[l], kv->v[l], kv->cap, kv->len, nullptr, nullptr,
                        batch, T, H, G, d, true, f.o)))
      return rc;
    if ((rc = mlp_tail(h, s, L, f, R))) return rc;
    for (int j = 0; j < n_taps; ++j)
      if (tap_ids[j] == l &&
          (rc = cast_rows(h, s, dt, f.x, (void*)byte_off(taps_out, (int64_t)j * R * D, dt), R * D)))
        return rc;
  }
  if ((rc = lm_head(h, s, f, f.x, R, h->w.g_f, 0, argmax_out, nullptr, 0, nullptr))) return rc;
  return advance_len(h, s, kv->len, nullptr, T, batch, kv->cap);
}

int dflash_selftest_wait(dflash_handle* h, int32_t which, int64_t limit_ns, dflash_stream_t s) {
  if (!h || (which != 0 && which != 1) || limit_ns < 1000 || limit_ns > 1000000000)
    return DFLASH_ERR_INVALID_ARG;
  return selftest_wait(h, (cudaStream_t)s, which, limit_ns);
}

int dflash_get_status(dflash_handle* h, dflash_stream_t st) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)st) != cudaSuccess) return DFLASH_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, h->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DFLASH_ERR_CUDA;
  cudaMemset(h->d_status, 0, sizeof(int));
  // a launch that gave up may have left tile counters mid-count
  if (v & ST_TIMEOUT) cudaMemset(h->d_counters, 0, kCounters * sizeof(int));
  if (v & ST_CAPACITY) return DFLASH_ERR_CAPACITY;
  if (v & ST_BOUNDS) return DFLASH_ERR_DEVICE_BOUNDS;
  if (v & ST_TIMEOUT) return DFLASH_ERR_DEVICE_TIMEOUT;
  return cudaGetLastError() == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

int dflash_timing_enable(dflash_handle* h, int on) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  h->timing = on != 0;
  return DFLASH_OK;
}

int dflash_timing_read(dflash_handle* h, int32_t kclass, double* total_ms, int64_t* launches) {
  if (!h || kclass < 0 || kclass >= DFLASH_K_NCLASS || !total_ms || !launches)
    return DFLASH_ERR_INVALID_ARG;
  if (!h->pending.empty()) {
    for (auto& t : h->pending) {
      float ms = 0.f;
      cudaEventSynchronize(t.b);
      cudaEventElapsedTime(&ms, t.a, t.b);
      h->ms[t.kclass] += ms;
      h->launches[t.kclass] += 1;
      h->free_events.push_back(t.a);
      h->free_events.push_back(t.b);
    }
    h->pending.clear();
  }
  *total_ms = h->ms[kclass];
  *launches = h->launches[kclass];
  h->ms[kclass] = 0;
  h->launches[kclass] = 0;
  return DFLASH_OK;
}

int dflash_chain_trace_enable(dflash_handle* h, int on) {
  if (!h) return DFLASH_ERR_INVALID_ARG;
  if (on && !h->d_trace) {
    if (cudaMalloc(&h->d_trace, (kChainTraceCols * kChainMaxPhases + kEvWords) *
                                    sizeof(unsigned long long)) != cudaSuccess) {
      h->d_trace = nullptr;
      return DFLASH_ERR_CUDA;
    }
    h->trace_phases = 0;
  } else if (!on && h->d_trace) {
    cudaDeviceSynchronize();
    cudaFree(h->d_trace);
    h->d_trace = nullptr;
  }
  return DFLASH_OK;
}

int dflash_chain_trace_read(dflash_handle* h, int64_t* out, int32_t n, int32_t* n_phases) {
  if (!h || !n_phases || n < 0 || (n > 0 && !out)) return DFLASH_ERR_INVALID_ARG;
  *n_phases = 0;
  if (!h->d_trace || h->trace_phases == 0) return DFLASH_OK;
  std::vector<unsigned long long> t(kChainTraceCols * kChainMaxPhases);
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(t.data(), h->d_trace, t.size() * sizeof(t[0]), cudaMemcpyDeviceToHost) !=
          cudaSuccess)
    return DFLASH_ERR_CUDA;
  const int np = h->trace_phases;
  for (int p = 0; p < np && p < n; ++p)
    for (int k = 0; k < kChainTraceCols; ++k) {
      const unsigned long long v = t[(size_t)k * kChainMaxPhases + p];
      out[kChainTraceCols * p + k] = v == ~0ull ? 0 : (int64_t)v;
    }
  *n_phases = np;
  return DFLASH_OK;
}

int dflash_chain_trace_events(dflash_handle* h, int64_t* out, int64_t n, int64_t* count) {
  if (!h || !count || n < 0 || (n > 0 && !out)) return DFLASH_ERR_INVALID_ARG;
  *count = 0;
  if (!h->d_trace || h->trace_phases == 0) return DFLASH_OK;
  const int64_t m = std::min<int64_t>(n, (int64_t)kEvWords);
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(out, h->d_trace + kChainTraceCols * kChainMaxPhases, m * sizeof(int64_t),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return DFLASH_ERR_CUDA;
  *count = m;
  return DFLASH_OK;
}

}  // extern "C"

namespace dflash {

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool make_tmap_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, int dtype,
                  bool swizzle128) {
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  }
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  const CUtensorMapDataType ty =
      dtype == DFLASH_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return g_encode(m, ty, 2, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace dflash
