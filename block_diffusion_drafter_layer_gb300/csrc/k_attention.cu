// Split-K attention of the draft block over [context cache ; block] (bf16).
//
// For one sequence b and one key/value head g the queries are the block's B
// rows of the H/G query heads that share g (at most 64 rows per query group);
// the keys are the L_b cached context entries followed by the block's own B
// rows, all visible (txtmix §6: full-attention draft layers are non-causal).
// A (b, g, query group) is a "unit".  Three launches:
//   attn_plan_kernel     reads the context lengths on the device and cuts
//                        every unit's keys into items of one common length (a
//                        multiple of 64 keys) chosen so that about AT_WAVES
//                        items fall on each resident CTA; it runs once per
//                        draft block, since the lengths do not change between
//                        layers;
//   attn_split_kernel    persistent CTAs (2 per SM) take the items
//                        round-robin: stream the item's keys in 64-key
//                        sub-chunks (cp.async, 3 stages), S = Q K^T and P V
//                        with warp-level bf16 MMA (fp32 accumulate), online
//                        softmax with the row max and sum reduced over quad
//                        shuffles, and write (max, sum, unnormalised output)
//                        per query row;
//   attn_combine_kernel  one warp per (unit, query row) merges the unit's
//                        items in key order and writes the bf16 output.
// Items depend only on the lengths of the batch, so results are
// deterministic.
#include "common.cuh"
#include "ptx.cuh"
#include "tc05.cuh"

// attention probabilities enter P V as a bf16 (hi, lo) pair (1) or as bf16 (0)
#ifndef DFLASH_AT_PLO
#define DFLASH_AT_PLO 1
#endif

namespace dflash {

using namespace ptx;

constexpr int AT_THREADS = 128;
constexpr int AT_KSUB = 64;              // keys per sub-chunk
constexpr int AT_STAGES = 3;             // cp.async pipeline depth of K/V sub-chunks
constexpr int AT_CTAS_PER_SM = 2;
constexpr int AT_WAVES = 3;              // items per persistent CTA, as a target
constexpr int AT_MIN_SUB = 4;            // sub-chunks per item, at least
constexpr int AT_MAX_ITEMS_UNIT = 128;   // items per unit, at most
constexpr int AT_DP = 132;               // floats per partial row: max, sum, 2 pad, 128 outputs
constexpr int AT_COMB_WARPS = 8;         // query rows per combine CTA

struct AttnItem {
  int unit, k0, k1, pad;   // keys [k0, k1) of the unit
};

struct AttnParams {
  const bf16* q;       // [batch*B, H*d]
  const bf16* kc;      // [batch_cap, G, cap, d]
  const bf16* vc;
  const bf16* kb;      // [batch*B, G*d] block keys
  const bf16* vb;
  bf16* o;             // [batch*B, H*d]
  const int32_t* len;  // [batch]
  int cap, B, H, G, rep, qgroups, units;
  float scale_log2;    // log2(e) / sqrt(d)
  int causal, window;  // the layer's mask: causal rows, a window of keys (0: none)
  const int* n_items;  // number of items (written by the plan)
  const AttnItem* items;
  const int* unit_begin;   // [units + 1] first item of each unit
  float* part;         // [max_items][64][AT_DP]
  int* status;
};

// Scratch region layout: header, unit offsets, items, partials.
struct AttnScratch {
  int* hdr;
  int* unit_begin;
  AttnItem* items;
  float* part;
};

static size_t r256(size_t x) { return (x + 255) & ~size_t(255); }

static int attn_units(const dflash_handle* h, int batch, int B) {
  const dflash_config& c = h->cfg;
  const int rep = c.n_heads / c.n_kv_heads, qgroups = (B * rep + 63) / 64;
  return batch * c.n_kv_heads * qgroups;
}
static int attn_slots(const dflash_handle* h) { return AT_CTAS_PER_SM * std::max(1, h->num_sms); }
// The plan cuts T sub-chunks into items of C >= T / (AT_WAVES * slots)
// sub-chunks each, so the items number at most AT_WAVES * slots + units.
static int64_t attn_max_items(const dflash_handle* h, int batch, int B) {
  return (int64_t)AT_WAVES * attn_slots(h) + attn_units(h, batch, B);
}
static AttnScratch attn_carve(float* scratch, int units, int64_t max_items) {
  char* p = reinterpret_cast<char*>(scratch);
  AttnScratch s;
  s.hdr = reinterpret_cast<int*>(p);
  p += 256;
  s.unit_begin = reinterpret_cast<int*>(p);
  p += r256((size_t)(units + 1) * sizeof(int));
  s.items = reinterpret_cast<AttnItem*>(p);
  p += r256((size_t)max_items * sizeof(AttnItem));
  s.part = reinterpret_cast<float*>(p);
  return s;
}

size_t attn_scratch_bytes(const dflash_handle* h, int batch, int B) {
  const int units = attn_units(h, batch, B);
  const int64_t mi = attn_max_items(h, batch, B);
  return 256 + r256((size_t)(units + 1) * sizeof(int)) + r256((size_t)mi * sizeof(AttnItem)) +
         (size_t)mi * 64 * AT_DP * sizeof(float) + 256;
}

// ---- plan: items of equal length over all units ----------------------------
__global__ void __launch_bounds__(256) attn_plan_kernel(const int32_t* len, int batch, int B,
                                                        int cap, int per_b, int slots, int cmul,
                                                        int max_items, int* hdr, int* unit_begin,
                                                        AttnItem* items, int* status) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ long long s_t[8];
  __shared__ int s_m[8], s_c, s_n;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  long long t = 0;
  int mx = 0;
  for (int b = tid; b < batch; b += blockDim.x) {
    const int L = len[b];
    if (L < 0 || L > cap) {
      atomicOr(status, ST_BOUNDS);
      continue;
    }
    const int ns = (L + B + AT_KSUB - 1) / AT_KSUB;
    t += ns;
    mx = max(mx, ns);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    t += __shfl_xor_sync(0xffffffffu, t, o);
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    s_t[warp] = t;
    s_m[warp] = mx;
  }
  __syncthreads();
  if (tid == 0) {
    long long T = 0;
    int M = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      T += s_t[w];
      M = max(M, s_m[w]);
    }
    T *= per_b;
    const long long cw = (T + (long long)AT_WAVES * slots - 1) / ((long long)AT_WAVES * slots);
    long long c = cw > AT_MIN_SUB ? cw : AT_MIN_SUB;
    const long long cm = (M + AT_MAX_ITEMS_UNIT - 1) / AT_MAX_ITEMS_UNIT;
    if (cm > c) c = cm;
    c = (c + cmul - 1) / cmul * cmul;   // whole sub-chunks of the kernel that takes the items
    const int C = (int)c;
    int n = 0;
    for (int b = 0; b < batch; ++b) {
      const int L = len[b];
      const bool ok = L >= 0 && L <= cap;
      const int ns = ok ? (L + B + AT_KSUB - 1) / AT_KSUB : 0;
      const int per = (ns + C - 1) / C;
      for (int j = 0; j < per_b; ++j) {
        unit_begin[b * per_b + j] = n;
        n += per;
      }
    }
    unit_begin[batch * per_b] = n;
    if (n > max_items) {   // cannot happen: C bounds the count
      atomicOr(status, ST_BOUNDS);
      n = 0;
    }
    hdr[0] = n;
    s_c = C;
    s_n = n;
  }
  __syncthreads();
  if (s_n == 0) return;
  const int C = s_c, units = batch * per_b;
  for (int u = tid; u < units; u += blockDim.x) {
    const int L = len[u / per_b];
    if (L < 0 || L > cap) continue;
    const int keys = L + B;
    const int i0 = unit_begin[u], i1 = unit_begin[u + 1];
    for (int i = i0; i < i1; ++i) {
      const int k0 = (i - i0) * C * AT_KSUB;
      items[i] = AttnItem{u, k0, min(keys, k0 + C * AT_KSUB), 0};
    }
  }
}

// smem tile of rows x DH bf16 (row = 2*DH bytes), 16-byte chunks XOR-swizzled
// by (row & 7) so 8 rows of one chunk column hit distinct banks.
template <int DH>
__device__ __forceinline__ uint32_t tile_off(int row, int chunk) {
  return (uint32_t)(row * (DH * 2) + ((chunk ^ (row & 7)) << 4));
}

// ---- the items: one partial softmax per (item, query row) --------------------
template <int DH>
__global__ void __launch_bounds__(AT_THREADS, AT_CTAS_PER_SM) attn_split_kernel(const AttnParams p) {
  constexpr int CH = DH / 8;               // 16-byte chunks per row
  constexpr int NT = DH / 8;               // n8 tiles of the output
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((128 - (smem_u32(smem_raw) & 127)) & 127);
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + 64 * DH * 2;
  const uint32_t sV0 = sK0 + AT_STAGES * AT_KSUB * DH * 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tg = lane & 3;
  pdl_launch_dependents();
  pdl_wait();
  const int n_items = *p.n_items;
  const int QM = p.B * p.rep;

  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const AttnItem item = p.items[it];
    const int u = item.unit;
    const int qg = u % p.qgroups, bg = u / p.qgroups;
    const int g = bg % p.G, b = bg / p.G;
    const int L = p.len[b];
    const int q0 = qg * 64;
    const int qrows = min(64, QM - q0);
    const int k_begin = item.k0, k_end = item.k1;
    // this thread's two query rows (tile rows warp * 16 + gq and + 8; block
    // row i at position L + i): keys [klo, khi) visible
    int klo[2], khi[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int qr = q0 + warp * 16 + gq + 8 * h;
      const int pq = L + (qr < QM ? qr % p.B : 0);
      klo[h] = p.window > 0 ? max(0, pq - p.window + 1) : 0;
      khi[h] = p.causal ? pq + 1 : k_end;
    }

    // ---- Q tile: row r = query (q0 + r) = head hh of the group, block row i
    for (int e = tid; e < 64 * CH; e += AT_THREADS) {
      const int r = e / CH, c = e - r * CH;
      const int qr = q0 + r;
      const bool ok = r < qrows;
      const int hh = ok ? qr / p.B : 0, i = ok ? qr - hh * p.B : 0;
      const bf16* src =
          p.q + (int64_t)(b * p.B + i) * (p.H * DH) + (int64_t)(g * p.rep + hh) * DH + c * 8;
      cp_async16(sQ + tile_off<DH>(r, c), ok ? src : p.q, ok);
    }
    const bf16* kcb = p.kc + ((int64_t)b * p.G + g) * p.cap * DH;
    const bf16* vcb = p.vc + ((int64_t)b * p.G + g) * p.cap * DH;
    const bf16* kbb = p.kb + (int64_t)b * p.B * (p.G * DH) + (int64_t)g * DH;
    const bf16* vbb = p.vb + (int64_t)b * p.B * (p.G * DH) + (int64_t)g * DH;
    auto load_kv = [&](int k0, int stage) {
      const uint32_t dk = sK0 + stage * AT_KSUB * DH * 2, dv = sV0 + stage * AT_KSUB * DH * 2;
      if (k0 + AT_KSUB <= min(L, k_end)) {
        // all 64 keys in the cache: the same (row, chunk) pairs as below with
        // the chunk fixed per thread and rows a constant stride apart
        constexpr int RSTEP = AT_THREADS / CH;
        const int c = tid % CH, r0 = tid / CH;
        const bf16* ks = kcb + (int64_t)(k0 + r0) * DH + c * 8;
        const bf16* vs = vcb + (int64_t)(k0 + r0) * DH + c * 8;
#pragma unroll
        for (int i = 0; i < AT_KSUB / RSTEP; ++i) {
          cp_async16(dk + tile_off<DH>(r0 + i * RSTEP, c), ks + (int64_t)i * RSTEP * DH, true);
          cp_async16(dv + tile_off<DH>(r0 + i * RSTEP, c), vs + (int64_t)i * RSTEP * DH, true);
        }
        return;
      }
      for (int e = tid; e < AT_KSUB * CH; e += AT_THREADS) {
        const int r = e / CH, c = e - r * CH;
        const int j = k0 + r;
        const bool ok = j < k_end;
        const bf16 *ks, *vs;
        if (j < L) {
          ks = kcb + (int64_t)j * DH + c * 8;
          vs = vcb + (int64_t)j * DH + c * 8;
        } else {
          const int jb = ok ? j - L : 0;
          ks = kbb + (int64_t)jb * (p.G * DH) + c * 8;
          vs = vbb + (int64_t)jb * (p.G * DH) + c * 8;
        }
        cp_async16(dk + tile_off<DH>(r, c), ok ? ks : kcb, ok);
        cp_async16(dv + tile_off<DH>(r, c), ok ? vs : vcb, ok);
      }
    };
    const int nsub = (k_end - k_begin + AT_KSUB - 1) / AT_KSUB;
    // prologue: the first AT_STAGES-1 sub-chunks (the Q tile rides in group 0)
#pragma unroll
    for (int st = 0; st < AT_STAGES - 1; ++st) {
      if (st < nsub) load_kv(k_begin + st * AT_KSUB, st);
      cp_async_commit();
    }

    const bool active = warp * 16 < qrows;
    uint32_t qa[DH / 16][4];
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

    for (int sc = 0; sc < nsub; ++sc) {
      const int stage = sc % AT_STAGES;
      // groups 0 .. sc + AT_STAGES - 2 are committed: sub-chunk sc has landed
      // once at most AT_STAGES - 2 remain in flight
      cp_async_wait<AT_STAGES - 2>();
      // all warps see sub-chunk sc and have finished sub-chunk sc - 1, whose
      // stage the next prefetch overwrites
      __syncthreads();
      const int pre = sc + AT_STAGES - 1;
      if (pre < nsub) load_kv(k_begin + pre * AT_KSUB, pre % AT_STAGES);
      cp_async_commit();
      if (sc == 0 && active) {
#pragma unroll
        for (int ks = 0; ks < DH / 16; ++ks) {
          const int row = warp * 16 + (lane & 15);
          const int ch = 2 * ks + (lane >> 4);
          ldsm_x4(sQ + tile_off<DH>(row, ch), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
        }
      }
      if (active) {
        const uint32_t sK = sK0 + stage * AT_KSUB * DH * 2, sV = sV0 + stage * AT_KSUB * DH * 2;
        const int kbase = k_begin + sc * AT_KSUB;
        // S = Q K^T for 64 keys: 8 n8 tiles
        float s[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < DH / 16; ++ks) {
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) {
            const int row = pp * 16 + (lane & 7) + ((lane >> 4) << 3);
            const int ch = 2 * ks + ((lane >> 3) & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(sK + tile_off<DH>(row, ch), b0, b1, b2, b3);
            mma_bf16_16816(s[2 * pp], qa[ks], b0, b1);
            mma_bf16_16816(s[2 * pp + 1], qa[ks], b2, b3);
          }
        }
        // online softmax over this sub-chunk (base-2 exponent, scale folded in);
        // plain: a bidirectional layer and all 64 keys inside the item, so
        // every key is visible and the visibility tests drop out
        const bool plain = !p.causal && p.window <= 0 && kbase + AT_KSUB <= k_end;
        float mnew[2] = {mrow[0], mrow[1]};
        if (plain) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              s[j][q] *= p.scale_log2;
              mnew[q >> 1] = fmaxf(mnew[q >> 1], s[j][q]);
            }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int key = kbase + j * 8 + 2 * tg + (q & 1);
              const bool vis = key < k_end && key >= klo[q >> 1] && key < khi[q >> 1];
              s[j][q] = vis ? s[j][q] * p.scale_log2 : -INFINITY;
              mnew[q >> 1] = fmaxf(mnew[q >> 1], s[j][q]);
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mnew[h] = fmaxf(mnew[h], __shfl_xor_sync(0xffffffffu, mnew[h], 1));
          mnew[h] = fmaxf(mnew[h], __shfl_xor_sync(0xffffffffu, mnew[h], 2));
        }
        float alpha[2], lsum[2] = {0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h) alpha[h] = (mrow[h] == -INFINITY) ? 0.f : exp2f(mrow[h] - mnew[h]);
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            // a row may see no key of this item yet (masked layers): weight 0
            const float e = (!plain && mnew[q >> 1] == -INFINITY) ? 0.f : exp2f(s[j][q] - mnew[q >> 1]);
            s[j][q] = e;
            lsum[q >> 1] += e;
          }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          lrow[h] = lrow[h] * alpha[h] + lsum[h];
          mrow[h] = mnew[h];
        }
        // once the running maxima settle alpha is exactly 1: skip the rescale
        if (!__all_sync(0xffffffffu, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            acc[j][0] *= alpha[0];
            acc[j][1] *= alpha[0];
            acc[j][2] *= alpha[1];
            acc[j][3] *= alpha[1];
          }
        }
        // O += P V with P as a bf16 pair hi + lo (hi = bf16(P), lo = bf16(P - hi):
        // P to about 16 bits) when DFLASH_AT_PLO, else hi alone; the row sum
        // above keeps fp32 P
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
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
          for (int np = 0; np < NT / 2; ++np) {
            const int row = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
            const int ch = np * 2 + (lane >> 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(sV + tile_off<DH>(row, ch), b0, b1, b2, b3);
            mma_bf16_16816(acc[2 * np], ph, b0, b1);
            mma_bf16_16816(acc[2 * np + 1], ph, b2, b3);
            if (DFLASH_AT_PLO) {
              mma_bf16_16816(acc[2 * np], pl, b0, b1);
              mma_bf16_16816(acc[2 * np + 1], pl, b2, b3);
            }
          }
        }
      }
    }
    cp_async_wait<0>();

    // ---- partial of this item: per query row (max, sum, unnormalised O) ----
    float* part = p.part + (int64_t)it * 64 * AT_DP;
    if (active) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 1);
        lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 2);
      }
      const int r0 = warp * 16 + gq, r1 = r0 + 8;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int col = j * 8 + 2 * tg;
        __stcg((float2*)&part[r0 * AT_DP + 4 + col], make_float2(acc[j][0], acc[j][1]));
        __stcg((float2*)&part[r1 * AT_DP + 4 + col], make_float2(acc[j][2], acc[j][3]));
      }
      if (tg == 0) {
        __stcg((float2*)&part[r0 * AT_DP], make_float2(mrow[0], lrow[0]));
        __stcg((float2*)&part[r1 * AT_DP], make_float2(mrow[1], lrow[1]));
      }
    }
    __syncthreads();
  }
}

// ---- combine: one warp per (unit, query row), items added in key order ------
template <int DH>
__global__ void __launch_bounds__(AT_COMB_WARPS * 32) attn_combine_kernel(const AttnParams p) {
  static_assert(DH == 128, "the combine maps 32 lanes x float4 onto a 128-wide row");
  __shared__ float wsm[AT_COMB_WARPS][AT_MAX_ITEMS_UNIT];
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = blockIdx.x * AT_COMB_WARPS + warp;
  const int u = gr >> 6, r = gr & 63;
  if (u >= p.units) return;
  const int qg = u % p.qgroups, bg = u / p.qgroups;
  const int g = bg % p.G, b = bg / p.G;
  const int q0 = qg * 64, qrows = min(64, p.B * p.rep - q0);
  if (r >= qrows) return;
  const int i0 = p.unit_begin[u], ns = p.unit_begin[u + 1] - i0;
  if (ns <= 0 || ns > AT_MAX_ITEMS_UNIT) return;   // no items: the plan flagged a bad length
  const float* base = p.part + ((int64_t)i0 * 64 + r) * AT_DP;
  const int64_t stride = 64 * AT_DP;
  float M = -INFINITY;
  for (int s = lane; s < ns; s += 32) M = fmaxf(M, __ldcg(base + s * stride));
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float lt = 0.f;
  for (int s = lane; s < ns; s += 32) {
    const float2 ml = __ldcg((const float2*)(base + s * stride));
    const float w = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
    wsm[warp][s] = w;
    lt += ml.y * w;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, o);
  __syncwarp();
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < ns; s0 += 8) {
    float4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int s = min(s0 + k, ns - 1);
      v[k] = __ldcg((const float4*)(base + s * stride + 4) + lane);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float w = (s0 + k < ns) ? wsm[warp][s0 + k] : 0.f;
      acc.x += v[k].x * w;
      acc.y += v[k].y * w;
      acc.z += v[k].z * w;
      acc.w += v[k].w * w;
    }
  }
  const float iv = 1.0f / lt;
  const int qr = q0 + r, hh = qr / p.B, i = qr - hh * p.B;
  bf16* dst = p.o + (int64_t)(b * p.B + i) * (p.H * DH) + (int64_t)(g * p.rep + hh) * DH + 4 * lane;
  __nv_bfloat162 t0 = __floats2bfloat162_rn(acc.x * iv, acc.y * iv);
  __nv_bfloat162 t1 = __floats2bfloat162_rn(acc.z * iv, acc.w * iv);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&t0);
  pk.y = *reinterpret_cast<uint32_t*>(&t1);
  *reinterpret_cast<uint2*>(dst) = pk;
}

// ---- the items on tcgen05 (blocks of 8, 16, 32 or 64 rows, d = 128) -----------
// One CTA per SM walks the items like attn_split_kernel and writes the same
// partials.  Per 128-key sub-chunk of an item: S = Q K^T on the tensor cores
// (M = 128 with the unit's query rows in rows 0-63, N = 128 keys, K = d) into
// one of three TMEM buffers; four softmax warps (TMEM lanes 0-63: a query row
// per thread, each key half in its own warp) take the row max over the
// sub-chunk, exchange it with the other half, and overwrite the S columns they
// have read with P as a bf16 pair (hi = bf16(p), lo = bf16(p - hi));
// O += P_hi V + P_lo V with A = P from TMEM and B = the V sub-chunk read
// MN-major from shared memory accumulates in TMEM.  The max used in the
// exponents moves only when a row's max rises by more than AT_TC_SLACK
// (log2), so O is rescaled rarely (p <= 2^8) and the softmax of a sub-chunk
// waits for the previous P V only then.  K/V sub-chunks of the cache (and
// the block's own rows, last) arrive by TMA in a 3-stage ring; V rows at
// positions >= len (stale cache memory) are zeroed before P V reads them.
// Warp 2 lane 0 issues the MMAs, warp 3 lane 0 the loads.
constexpr int AT_TC_THREADS = 192;
constexpr int AT_TC_KSUB = 128;
constexpr int AT_TC_STAGES = 3;
constexpr int AT_TC_HALF = 16384;                   // 128 rows x 64 d (one 64-d half)
constexpr int AT_TC_OFF_KV = 2 * AT_TC_HALF;        // after the Q tile
constexpr int AT_TC_STAGE = 4 * AT_TC_HALF;         // K (two halves), then V
constexpr int AT_TC_OFF_BAR = AT_TC_OFF_KV + AT_TC_STAGES * AT_TC_STAGE;
// [3][2 halves][64 rows] floats: the row maxima of sub-chunks with S buffer
// 0 and 1, then the row sums at the end of an item
constexpr int AT_TC_OFF_RED = AT_TC_OFF_BAR + 128;
constexpr int AT_TC_SMEM = AT_TC_OFF_RED + 3 * 2 * 64 * 4 + 1024;
static_assert(AT_TC_SMEM <= 232448, "shared memory per CTA");
// TMEM columns: S / P (three buffers: an S MMA into a buffer waits for the
// P V that read the buffer's P, issued two sub-chunks earlier), O
constexpr uint32_t AT_TM_S = 0, AT_TM_O = 384, AT_TM_COLS = 512;
constexpr float AT_TC_SLACK = 8.f;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// (lo, hi) -> bf16x2 with lo in the low half, round to nearest even
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

struct AttnTcParams {
  AttnParams a;
  CUtensorMap qmap;    // q [R, H d]: box 64 x B rows
  CUtensorMap kmap;    // the K cache as [kv_batch G cap, d]: box 64 x 128
  CUtensorMap vmap;
  CUtensorMap kbmap;   // the block's K [R, G d]: box 64 x 16
  CUtensorMap vbmap;
  int nb;              // block rows loaded per unit: max(16, B)
};

// Geometry of an item: unit (b, g, query rows q0 ..), keys [k0, k1); nc cache
// sub-chunks over [k0, min(k1, L)), then one block sub-chunk if k1 > L.
struct TcGeo {
  int b, g, q0, qrows, L, k0, k1, nc, nsub;
};
__device__ __forceinline__ TcGeo tc_geo(const AttnParams& p, const AttnItem& it) {
  TcGeo q;
  const int u = it.unit;
  const int qg = u % p.qgroups, bg = u / p.qgroups;
  q.g = bg % p.G;
  q.b = bg / p.G;
  q.q0 = qg * 64;
  q.qrows = min(64, p.B * p.rep - q.q0);
  q.L = p.len[q.b];
  q.k0 = it.k0;
  q.k1 = it.k1;
  const int ce = min(q.k1, q.L);
  q.nc = ce > q.k0 ? (ce - q.k0 + AT_TC_KSUB - 1) / AT_TC_KSUB : 0;
  q.nsub = q.nc + (q.k1 > q.L ? 1 : 0);
  return q;
}

__global__ void __launch_bounds__(AT_TC_THREADS, 1) attn_tc_kernel(const __grid_constant__ AttnTcParams tp) {
  const AttnParams& p = tp.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sQ = smem_u32(smem), sKV = sQ + AT_TC_OFF_KV;
  const uint32_t bar = sQ + AT_TC_OFF_BAR;
  // barriers: kv_full[3], kv_empty[3], q_full, q_empty, s_full[3] and
  // pv_done[3] (per S / P buffer), p_full
  const uint32_t b_kvf = bar, b_kve = bar + 24, b_qf = bar + 48, b_qe = bar + 56, b_sf = bar + 64,
                 b_pf = bar + 88, b_pv = bar + 96;
  volatile uint32_t* tmem_slot = (volatile uint32_t*)(smem + AT_TC_OFF_BAR + 120);
  volatile int* abort_flag = (volatile int*)(smem + AT_TC_OFF_BAR + 124);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < AT_TC_STAGES; ++s) {
      mbar_init(b_kvf + 8 * s, 1);
      mbar_init(b_kve + 8 * s, 1);
    }
    mbar_init(b_qf, 1);
    mbar_init(b_qe, 1);
    for (int b = 0; b < 3; ++b) {
      mbar_init(b_sf + 8 * b, 1);
      mbar_init(b_pv + 8 * b, 1);
    }
    mbar_init(b_pf, 128);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32((const void*)tmem_slot)),
                 "r"(AT_TM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();
  const int n_items = *p.n_items;
  const int nb = tp.nb;
  auto fail = [&]() {
    atomicOr(p.status, ST_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 3) {
    if (lane == 0) {
      // ---- loads ----------------------------------------------------------------
      int qn = 0, ni = 0;
      for (int it = blockIdx.x; it < n_items && !*abort_flag; it += gridDim.x, ++ni) {
        const TcGeo q = tc_geo(p, p.items[it]);
        // the Q tile: rows hh * B - q0 .. of the heads hh that hold rows q0 .. q0 + qrows
        if (ni > 0 && !mbar_wait(b_qe, (ni - 1) & 1)) { fail(); break; }
        const int h0 = q.q0 / p.B, h1 = (q.q0 + q.qrows - 1) / p.B;
        mbar_arrive_expect_tx(b_qf, (uint32_t)(2 * (h1 - h0 + 1) * p.B * 128));
        for (int hh = h0; hh <= h1; ++hh)
          for (int h = 0; h < 2; ++h)
            tma_load_2d(sQ + h * AT_TC_HALF + (hh * p.B - q.q0) * 128, &tp.qmap, b_qf,
                        (q.g * p.rep + hh) * 128 + h * 64, q.b * p.B, policy_evict_first());
        for (int j = 0; j < q.nsub; ++j) {
          const int qq = qn + j, st = qq % AT_TC_STAGES, use = qq / AT_TC_STAGES;
          if (use > 0 && !mbar_wait(b_kve + 8 * st, (use - 1) & 1)) { fail(); break; }
          const uint32_t dK = sKV + st * AT_TC_STAGE, dV = dK + 2 * AT_TC_HALF;
          const uint32_t fb = b_kvf + 8 * st;
          if (j < q.nc) {
            const int key0 = q.k0 + j * AT_TC_KSUB;
            const int row = (q.b * p.G + q.g) * p.cap + key0;
            mbar_arrive_expect_tx(fb, 4 * AT_TC_HALF);
            for (int h = 0; h < 2; ++h) {
              tma_load_2d(dK + h * AT_TC_HALF, &tp.kmap, fb, h * 64, row, policy_evict_first());
              tma_load_2d(dV + h * AT_TC_HALF, &tp.vmap, fb, h * 64, row, policy_evict_first());
            }
          } else {
            mbar_arrive_expect_tx(fb, (uint32_t)(4 * nb * 128));
            for (int i = 0; i < nb; i += 16)
              for (int h = 0; h < 2; ++h) {
                tma_load_2d(dK + h * AT_TC_HALF + i * 128, &tp.kbmap, fb, q.g * 128 + h * 64,
                            q.b * p.B + i, policy_evict_first());
                tma_load_2d(dV + h * AT_TC_HALF + i * 128, &tp.vbmap, fb, q.g * 128 + h * 64,
                            q.b * p.B + i, policy_evict_first());
              }
          }
        }
        qn += q.nsub;
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    if (lane == 0) {
      // ---- MMAs -------------------------------------------------------------------
      int qn = 0, ni = 0;
      auto issue_s = [&](const TcGeo& q, int j) -> bool {
        const int qq = qn + j, st = qq % AT_TC_STAGES, sb = qq % 3;
        // the P V of sub-chunk qq - 3 read this buffer's P: done before S overwrites it
        if (qq >= 3 && !mbar_wait(b_pv + 8 * sb, (qq / 3 - 1) & 1)) return false;
        if (!mbar_wait(b_kvf + 8 * st, (qq / AT_TC_STAGES) & 1)) return false;
        tc_fence_after();
        const int n = j < q.nc ? AT_TC_KSUB : nb;
        const uint32_t idesc = idesc_bf16_f32(128, n);
        const uint32_t dK = sKV + st * AT_TC_STAGE;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma(tmem + AT_TM_S + sb * 128, sdesc_sw128(sQ + (kk >> 2) * AT_TC_HALF + (kk & 3) * 32),
                 sdesc_sw128(dK + (kk >> 2) * AT_TC_HALF + (kk & 3) * 32), idesc, kk > 0);
        tc_commit(b_sf + 8 * sb);
        return true;
      };
      for (int it = blockIdx.x; it < n_items && !*abort_flag; it += gridDim.x, ++ni) {
        const TcGeo q = tc_geo(p, p.items[it]);
        if (!mbar_wait(b_qf, ni & 1)) { fail(); break; }
        tc_fence_after();
        bool ok = true;
        for (int j = 0; ok && j < q.nsub && j < 2; ++j) ok = issue_s(q, j);
        if (ok && q.nsub <= 2) tc_commit(b_qe);
        for (int j = 0; ok && j < q.nsub; ++j) {
          const int qq = qn + j, st = qq % AT_TC_STAGES;
          if (!mbar_wait(b_pf, qq & 1)) { ok = false; break; }
          tc_fence_after();
          const int n = j < q.nc ? AT_TC_KSUB : nb;
          const uint32_t idesc = idesc_bf16_f32_bmn(128, 128);
          const uint32_t dV = sKV + st * AT_TC_STAGE + 2 * AT_TC_HALF;
          // P of keys 32c .. 32c + 31: hi in S columns 32c .. 32c + 15, lo in the next 16
          const uint32_t pb = tmem + AT_TM_S + (qq % 3) * 128;
          for (int ks = 0; ks < n / 16; ++ks) {
            const uint64_t vd = sdesc_sw128_lbo(dV + ks * 2048, AT_TC_HALF, 1024);
            const uint32_t pa = pb + 32 * (ks >> 1) + 8 * (ks & 1);
            tc_mma_ts(tmem + AT_TM_O, pa, vd, idesc, (j > 0 || ks > 0) ? 1u : 0u);
            tc_mma_ts(tmem + AT_TM_O, pa + 16, vd, idesc, 1u);
          }
          tc_commit(b_kve + 8 * st);
          tc_commit(b_pv + 8 * (qq % 3));
          if (j + 2 < q.nsub) {
            ok = issue_s(q, j + 2);
            if (ok && j + 2 == q.nsub - 1) tc_commit(b_qe);
          }
        }
        if (!ok) { fail(); break; }
        qn += q.nsub;
      }
    }
    __syncwarp();
  } else {
    // ---- softmax and partials: warps 0, 1 (keys 0-63 of a sub-chunk) and 4, 5
    // (keys 64-127); thread = query row r of the tile (TMEM lane r) ----------
    const int kh = warp >> 2;                        // key half
    const int r = (warp & 1) * 32 + lane;
    const int st_tid = kh * 64 + r;                  // 0 .. 127 over the four warps
    const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
    float* red = (float*)(smem + AT_TC_OFF_RED);     // [3][2][64]
    // After a timed-out wait the warps go on without waiting (results are
    // void, the status says so) so that all four meet at every named barrier.
    int qn = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
      const TcGeo q = tc_geo(p, p.items[it]);
      const bool row_ok = r < q.qrows;
      const int qr = q.q0 + (row_ok ? r : 0), i = qr % p.B;
      const int pq = q.L + i;
      const int klo = p.window > 0 ? max(0, pq - p.window + 1) : 0;
      const int khi = p.causal ? min(pq + 1, q.k1) : q.k1;
      const int lo = max(q.k0, klo);   // visible keys of this row in the item: [lo, khi)
      float m_use = -INFINITY, l = 0.f;
      for (int j = 0; j < q.nsub; ++j) {
        const int qq = qn + j, sb = qq & 1, tb = qq % 3;   // exchange buffer, S / P buffer
        const bool cache = j < q.nc;
        const int key0 = cache ? q.k0 + j * AT_TC_KSUB : q.L;
        const int n = cache ? AT_TC_KSUB : nb;
        // this row's visible columns of the sub-chunk: [vlo, vhi)
        const int lim = cache ? q.L : q.L + p.B;
        const int vlo = row_ok ? max(lo - key0, 0) : 0;
        const int vhi = row_ok ? max(min(min(khi, lim) - key0, n), vlo) : 0;
        const int c0 = kh * 64;   // this warp's columns c0 .. c0 + 63 (those below n)
        const uint32_t sbuf = tmem + lanes + AT_TM_S + tb * 128;
        if (ok) ok = __all_sync(0xffffffffu, !*abort_flag && mbar_wait(b_sf + 8 * tb, (qq / 3) & 1, 4000000000ull));
        tc_fence_after();
        // pass 1: the row max over this half's visible keys (columns at or
        // past n are stale and invisible)
        float mx = -INFINITY;
        float v[2][32];
        if (c0 < n) {
          tc_ld64(sbuf + c0, &v[0][0]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int cb = c0 + 32 * h;
            if (vlo <= cb && vhi >= cb + 32) {
              float m2 = v[h][0];
#pragma unroll
              for (int k = 1; k < 32; ++k) m2 = fmaxf(m2, v[h][k]);
              mx = fmaxf(mx, m2);
            } else {
#pragma unroll
              for (int k = 0; k < 32; ++k)
                if (cb + k >= vlo && cb + k < vhi) mx = fmaxf(mx, v[h][k]);
            }
          }
        }
        red[(sb * 2 + kh) * 64 + r] = mx;
        named_bar(1, 128);
        mx = fmaxf(mx, red[(sb * 2 + (kh ^ 1)) * 64 + r]);
        const float mnew = mx == -INFINITY ? m_use : fmaxf(m_use, mx * p.scale_log2);
        const bool resc = mnew > m_use + AT_TC_SLACK || (m_use == -INFINITY && mnew > -INFINITY);
        float alpha = 1.f;
        if (resc) {
          alpha = m_use == -INFINITY ? 0.f : ex2_approx(m_use - mnew);
          m_use = mnew;
        }
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
          // O holds every earlier sub-chunk's P V: rescale this half of its columns
          if (ok) ok = __all_sync(0xffffffffu, mbar_wait(b_pv + 8 * ((qq - 1) % 3), ((qq - 1) / 3) & 1, 4000000000ull));
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            float o[32];
            tc_ld32(tmem + lanes + AT_TM_O + kh * 64 + c * 32, o);
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] *= alpha;
            tc_st32(tmem + lanes + AT_TM_O + kh * 64 + c * 32, o);
          }
        }
        l *= alpha;
        // pass 2: p = 2^(s * scale - m_use) for visible keys as (hi, lo) bf16
        // pairs, over the S columns just read
        const float sc = p.scale_log2, nm = m_use == -INFINITY ? 0.f : -m_use;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int cb = c0 + 32 * h;
          if (cb < n) {
            const bool all = vlo <= cb && vhi >= cb + 32 && m_use > -INFINITY;
            uint32_t ph[16], pl[16];
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              float e0 = ex2_approx(fmaf(v[h][k], sc, nm));
              float e1 = ex2_approx(fmaf(v[h][k + 1], sc, nm));
              if (!all) {
                const bool m0 = m_use > -INFINITY && cb + k >= vlo && cb + k < vhi;
                const bool m1 = m_use > -INFINITY && cb + k + 1 >= vlo && cb + k + 1 < vhi;
                e0 = m0 ? e0 : 0.f;
                e1 = m1 ? e1 : 0.f;
              }
              l += e0 + e1;
              const uint32_t hi = bf16x2_rn(e0, e1);
              const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xffff0000u);
              ph[k >> 1] = hi;
              pl[k >> 1] = bf16x2_rn(e0 - h0, e1 - h1);
            }
            // columns 32c .. 32c + 15 take hi of keys 32c .. 32c + 31 (two per column),
            // the next 16 columns lo
            tc_st16(sbuf + cb, ph);
            tc_st16(sbuf + cb + 16, pl);
          }
        }
        // V rows at positions >= len in a cache sub-chunk: stale memory, zeroed
        if (cache && key0 + AT_TC_KSUB > q.L) {
          const int st = qq % AT_TC_STAGES;
          if (ok) ok = __all_sync(0xffffffffu, mbar_wait(b_kvf + 8 * st, (qq / AT_TC_STAGES) & 1));
          const int z0 = max(0, q.L - key0);
          uint8_t* dV = smem + AT_TC_OFF_KV + st * AT_TC_STAGE + 2 * AT_TC_HALF;
          for (int e = st_tid; e < (AT_TC_KSUB - z0) * 16; e += 128) {
            const int row = z0 + (e >> 4), c16 = e & 15;
            *(uint4*)(dV + (c16 >> 3) * AT_TC_HALF + row * 128 + (c16 & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(b_pf);
      }
      qn += q.nsub;
      // the item's partial: (max, sum, unnormalised O) of this row; each half
      // writes its 64 columns of O, half 0 the row's (max, sum of both halves)
      red[(4 + kh) * 64 + r] = l;
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(b_pv + 8 * ((qn - 1) % 3), ((qn - 1) / 3) & 1, 4000000000ull));
      tc_fence_after();
      named_bar(1, 128);
      float* part = p.part + ((int64_t)it * 64 + r) * AT_DP;
      {
        float o[64];
        tc_ld64(tmem + lanes + AT_TM_O + kh * 64, o);
        if (row_ok) {
#pragma unroll
          for (int k = 0; k < 64; k += 4)
            __stcg((float4*)&part[4 + kh * 64 + k], make_float4(o[k], o[k + 1], o[k + 2], o[k + 3]));
        }
      }
      if (row_ok && kh == 0) __stcg((float2*)part, make_float2(m_use, l + red[5 * 64 + r]));
      tc_fence_before();
      named_bar(1, 128);   // the sums are read before the next item writes them
    }
    if (!ok) fail();
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) {
    // loads or MMAs may still be in flight: let them land (bounded) before
    // the shared memory and TMEM are released
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 200000ull) __nanosleep(1000);
  }
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(AT_TM_COLS)
                 : "memory");
  }
}

bool attn_fast_ok(const dflash_handle* h, int B) {
  const dflash_config& c = h->cfg;
  return c.dtype == DFLASH_BF16 && c.head_dim == 128 && h->num_sms > 0 && B >= 1;
}

static void pdl_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, dim3 grid, dim3 block,
                       size_t smem, cudaStream_t s) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = grid;
  cfg->blockDim = block;
  cfg->dynamicSmemBytes = smem;
  cfg->stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
}

// The tcgen05 items kernel: bf16, d = 128, blocks of 8, 16, 32 or 64 rows
// (whole 8-row groups per query head in the 64-row tile).
#ifndef DFLASH_AT_TC
#define DFLASH_AT_TC 1
#endif
static bool attn_tc_ok(const dflash_handle* h, int B) {
  const dflash_config& c = h->cfg;
  return DFLASH_AT_TC && c.dtype == DFLASH_BF16 && c.head_dim == 128 &&
         (B == 8 || B == 16 || B == 32 || B == 64) && h->num_sms > 0;
}

int attn_plan(dflash_handle* h, cudaStream_t s, const int32_t* len, int cap, int batch, int B,
              float* scratch) {
  const dflash_config& c = h->cfg;
  const int rep = c.n_heads / c.n_kv_heads, qgroups = (B * rep + 63) / 64;
  const int units = attn_units(h, batch, B);
  const int64_t mi = attn_max_items(h, batch, B);
  if (mi > 0x7fffffff || (int64_t)units * 64 > 0x7fffffff) return DFLASH_ERR_SHAPE;
  const AttnScratch sc = attn_carve(scratch, units, mi);
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  pdl_config(&cfg, attr, dim3(1), dim3(256), 0, s);
  Timer t;
  launch_begin(h, DFLASH_K_ATTENTION, s, &t);
  // the tcgen05 kernel: one CTA per SM, items of whole 128-key sub-chunks
  const bool tc = attn_tc_ok(h, B);
  cudaLaunchKernelEx(&cfg, attn_plan_kernel, len, batch, B, cap, c.n_kv_heads * qgroups,
                     tc ? h->num_sms : attn_slots(h), tc ? 2 : 1, (int)mi, sc.hdr, sc.unit_begin,
                     sc.items, h->d_status);
  return launch_end(h, s, &t);
}

int attention_fast(dflash_handle* h, cudaStream_t s, const void* q, const void* kc, const void* vc,
                   int cap, int kv_batch, const int32_t* len, const void* kb, const void* vb,
                   int batch, int B, void* o, float* scratch, int causal, int window) {
  const dflash_config& c = h->cfg;
  constexpr int DH = 128;
  const int units = attn_units(h, batch, B);
  const int64_t mi = attn_max_items(h, batch, B);
  const AttnScratch sc = attn_carve(scratch, units, mi);
  AttnParams p;
  p.q = (const bf16*)q;
  p.kc = (const bf16*)kc;
  p.vc = (const bf16*)vc;
  p.kb = (const bf16*)kb;
  p.vb = (const bf16*)vb;
  p.o = (bf16*)o;
  p.len = len;
  p.cap = cap;
  p.B = B;
  p.causal = causal, p.window = window;
  p.H = c.n_heads;
  p.G = c.n_kv_heads;
  p.rep = c.n_heads / c.n_kv_heads;
  p.qgroups = (B * p.rep + 63) / 64;
  p.units = units;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)DH);
  p.n_items = sc.hdr;
  p.items = sc.items;
  p.unit_begin = sc.unit_begin;
  p.part = sc.part;
  p.status = h->d_status;
  if (attn_tc_ok(h, B)) {
    AttnTcParams tp;
    memset(&tp, 0, sizeof(tp));
    tp.a = p;
    tp.nb = std::max(16, B);
    const uint64_t Hd = (uint64_t)p.H * DH, Gd = (uint64_t)p.G * DH, R = (uint64_t)batch * B;
    if (!make_tmap_2d(&tp.qmap, q, Hd, R, Hd * 2, 64, (uint32_t)B) ||
        !make_tmap_2d(&tp.kmap, kc, DH, (uint64_t)kv_batch * p.G * cap, DH * 2, 64, AT_TC_KSUB) ||
        !make_tmap_2d(&tp.vmap, vc, DH, (uint64_t)kv_batch * p.G * cap, DH * 2, 64, AT_TC_KSUB) ||
        !make_tmap_2d(&tp.kbmap, kb, Gd, R, Gd * 2, 64, 16) ||
        !make_tmap_2d(&tp.vbmap, vb, Gd, R, Gd * 2, 64, 16))
      return DFLASH_ERR_CUDA;
    static bool tc_attr = false;
    if (!tc_attr) {
      if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               AT_TC_SMEM) != cudaSuccess)
        return DFLASH_ERR_CUDA;
      tc_attr = true;
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    pdl_config(&cfg, attr, dim3((unsigned)std::min<int64_t>(mi, h->num_sms)), dim3(AT_TC_THREADS),
               AT_TC_SMEM, s);
    Timer t;
    launch_begin(h, DFLASH_K_ATTENTION, s, &t);
    cudaLaunchKernelEx(&cfg, attn_tc_kernel, tp);
    int rc = launch_end(h, s, &t);
    if (rc) return rc;
    const int cgrid = (units * 64 + AT_COMB_WARPS - 1) / AT_COMB_WARPS;
    pdl_config(&cfg, attr, dim3(cgrid), dim3(AT_COMB_WARPS * 32), 0, s);
    launch_begin(h, DFLASH_K_ATTENTION, s, &t);
    cudaLaunchKernelEx(&cfg, attn_combine_kernel<DH>, p);
    return launch_end(h, s, &t);
  }
  // Q + AT_STAGES x (K, V) sub-chunks
  const size_t smem = (size_t)(64 + 2 * AT_STAGES * AT_KSUB) * DH * 2 + 128;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attn_split_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return DFLASH_ERR_CUDA;
    attr_set = true;
  }
  const int grid = (int)std::min<int64_t>(mi, attn_slots(h));
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  pdl_config(&cfg, attr, dim3(grid), dim3(AT_THREADS), smem, s);
  Timer t;
  launch_begin(h, DFLASH_K_ATTENTION, s, &t);
  cudaLaunchKernelEx(&cfg, attn_split_kernel<DH>, p);
  int rc = launch_end(h, s, &t);
  if (rc) return rc;
  const int cgrid = (units * 64 + AT_COMB_WARPS - 1) / AT_COMB_WARPS;
  pdl_config(&cfg, attr, dim3(cgrid), dim3(AT_COMB_WARPS * 32), 0, s);
  launch_begin(h, DFLASH_K_ATTENTION, s, &t);
  cudaLaunchKernelEx(&cfg, attn_combine_kernel<DH>, p);
  return launch_end(h, s, &t);
}

}  // namespace dflash
