// Split-K attention of the draft block over [context cache ; block] (bf16).
//
// For one sequence b and one key/value head g, the queries are the block's
// B rows of the H/G query heads that share g (B * H/G <= 64 rows per CTA
// group); the keys are the L_b cached context entries followed by the
// block's own B rows, all visible (txtmix §6: full-attention draft layers
// are non-causal).  The key axis is cut into fixed splits by absolute key
// index, one CTA per (split, g, b): the CTA streams its keys in 64-key
// sub-chunks (cp.async, double-buffered), computes S = Q K^T and P V with
// warp-level bf16 MMA (fp32 accumulate), and keeps a running max and sum
// per query row (online softmax, row max / sum reduced with quad shuffles).
// The probabilities enter the PV product as a bf16 pair (hi + lo) so they
// carry ~16 bits.  Each CTA writes (max, sum, unnormalised output) per row;
// the CTA that finishes a (b, g) last combines the splits in split order.
// Splits depend only on key positions, so a row's result does not depend on
// the batch or block size around it.
#include "common.cuh"
#include "ptx.cuh"

namespace dflash {

using namespace ptx;

constexpr int AT_THREADS = 128;
constexpr int AT_KSUB = 64;   // keys per sub-chunk
constexpr int AT_MAX_SPLITS = 128;   // splits per (b, g); bounds the combine's shared memory
constexpr int AT_MIN_SPLIT = 256;    // keys per split unless that leaves too few CTAs
constexpr int AT_STAGES = 3;         // cp.async pipeline depth of K/V sub-chunks

struct AttnParams {
  const bf16* q;       // [batch*B, H*d]
  const bf16* kc;      // [batch_cap, G, cap, d]
  const bf16* vc;
  const bf16* kb;      // [batch*B, G*d] block keys
  const bf16* vb;
  bf16* o;             // [batch*B, H*d]
  const int32_t* len;  // [batch]
  int cap, B, H, G, rep, split;
  float scale_log2;    // log2(e) / sqrt(d)
  float* part;         // [batch, G, qgroups, nsplit_max, 64, d + 4]
  int* counters;       // [batch * G * qgroups]
  int nsplit_max, qgroups;
  int* status;
};

// smem tile of rows x DH bf16 (row = 2*DH bytes), 16-byte chunks XOR-swizzled
// by (row & 7) so 8 rows of one chunk column hit distinct banks.
template <int DH>
__device__ __forceinline__ uint32_t tile_off(int row, int chunk) {
  return (uint32_t)(row * (DH * 2) + ((chunk ^ (row & 7)) << 4));
}

template <int DH>
__global__ void __launch_bounds__(AT_THREADS, 2) attn_split_kernel(const AttnParams p) {
  constexpr int CH = DH / 8;               // 16-byte chunks per row
  constexpr int NT = DH / 8;               // n8 tiles of the output
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((128 - (smem_u32(smem_raw) & 127)) & 127);
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + 64 * DH * 2;
  const uint32_t sV0 = sK0 + AT_STAGES * AT_KSUB * DH * 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, g = blockIdx.y;
  const int b = blockIdx.z / p.qgroups, qg = blockIdx.z - b * p.qgroups;
  pdl_launch_dependents();
  pdl_wait();

  const int L = p.len[b];
  const int nk = L + p.B;
  const int nsplit = (nk + p.split - 1) / p.split;
  if (split >= nsplit) return;
  if (L < 0 || L > p.cap || nsplit > p.nsplit_max) {
    if (tid == 0) atomicOr(p.status, ST_BOUNDS);
    return;
  }
  const int QM = p.B * p.rep;                 // query rows of this (b, g)
  const int q0 = qg * 64;
  const int qrows = min(64, QM - q0);
  const int k_begin = split * p.split, k_end = min(nk, k_begin + p.split);

  // ---- Q tile: row r = query (q0 + r) = head hh of the group, block row i
  for (int e = tid; e < 64 * CH; e += AT_THREADS) {
    const int r = e / CH, c = e - r * CH;
    const int qr = q0 + r;
    const bool ok = r < qrows;
    const int hh = ok ? qr / p.B : 0, i = ok ? qr - hh * p.B : 0;
    const bf16* src = p.q + (int64_t)(b * p.B + i) * (p.H * DH) + (int64_t)(g * p.rep + hh) * DH + c * 8;
    cp_async16(sQ + tile_off<DH>(r, c), ok ? src : p.q, ok);
  }
  const bf16* kcb = p.kc + ((int64_t)b * p.G + g) * p.cap * DH;
  const bf16* vcb = p.vc + ((int64_t)b * p.G + g) * p.cap * DH;
  const bf16* kbb = p.kb + (int64_t)b * p.B * (p.G * DH) + (int64_t)g * DH;
  const bf16* vbb = p.vb + (int64_t)b * p.B * (p.G * DH) + (int64_t)g * DH;
  auto load_kv = [&](int k0, int stage) {
    const uint32_t dk = sK0 + stage * AT_KSUB * DH * 2, dv = sV0 + stage * AT_KSUB * DH * 2;
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

  const int gq = lane >> 2, tg = lane & 3;
  const bool active = warp * 16 < qrows;
  uint32_t qa[DH / 16][4];
  float acc[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

  for (int sc = 0; sc < nsub; ++sc) {
    const int stage = sc % AT_STAGES;
    const int pre = sc + AT_STAGES - 1;
    if (pre < nsub) load_kv(k_begin + pre * AT_KSUB, pre % AT_STAGES);
    cp_async_commit();
    cp_async_wait<AT_STAGES - 1>();
    __syncthreads();
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
      // online softmax over this sub-chunk (base-2 exponent, scale folded in)
      float mnew[2] = {mrow[0], mrow[1]};
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int key = kbase + j * 8 + 2 * tg + (q & 1);
          s[j][q] = (key < k_end) ? s[j][q] * p.scale_log2 : -INFINITY;
          mnew[q >> 1] = fmaxf(mnew[q >> 1], s[j][q]);
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
          const float e = exp2f(s[j][q] - mnew[q >> 1]);
          s[j][q] = e;
          lsum[q >> 1] += e;
        }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        lrow[h] = lrow[h] * alpha[h] + lsum[h];
        mrow[h] = mnew[h];
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        acc[j][0] *= alpha[0];
        acc[j][1] *= alpha[0];
        acc[j][2] *= alpha[1];
        acc[j][3] *= alpha[1];
      }
      // O += P V, P as bf16 hi + lo
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t ph[4], pl[4];
        const float* s0 = s[2 * kk];
        const float* s1 = s[2 * kk + 1];
        const float v[8] = {s0[0], s0[1], s0[2], s0[3], s1[0], s1[1], s1[2], s1[3]};
        float hi[8], lo[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          hi[q] = __bfloat162float(__float2bfloat16_rn(v[q]));
          lo[q] = v[q] - hi[q];
        }
        ph[0] = pack_bf16(hi[0], hi[1]);
        ph[1] = pack_bf16(hi[2], hi[3]);
        ph[2] = pack_bf16(hi[4], hi[5]);
        ph[3] = pack_bf16(hi[6], hi[7]);
        pl[0] = pack_bf16(lo[0], lo[1]);
        pl[1] = pack_bf16(lo[2], lo[3]);
        pl[2] = pack_bf16(lo[4], lo[5]);
        pl[3] = pack_bf16(lo[6], lo[7]);
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          const int row = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int ch = np * 2 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sV + tile_off<DH>(row, ch), b0, b1, b2, b3);
          mma_bf16_16816(acc[2 * np], ph, b0, b1);
          mma_bf16_16816(acc[2 * np + 1], ph, b2, b3);
          mma_bf16_16816(acc[2 * np], pl, b0, b1);
          mma_bf16_16816(acc[2 * np + 1], pl, b2, b3);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // ---- partial of this split: per query row (max, sum, unnormalised O) ------
  const int DP = DH + 4;   // (max, sum, 2 pad, output) keeps the output 16-byte aligned
  const int bgq = (b * p.G + g) * p.qgroups + qg;
  float* part = p.part + ((int64_t)bgq * p.nsplit_max + split) * 64 * DP;
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
      *(float2*)&part[r0 * DP + 4 + col] = make_float2(acc[j][0], acc[j][1]);
      *(float2*)&part[r1 * DP + 4 + col] = make_float2(acc[j][2], acc[j][3]);
    }
    if (tg == 0) {
      part[r0 * DP] = mrow[0];
      part[r0 * DP + 1] = lrow[0];
      part[r1 * DP] = mrow[1];
      part[r1 * DP + 1] = lrow[1];
    }
  }
  __threadfence();
  __syncthreads();
  __shared__ int is_last;
  if (tid == 0) {
    const int old = atomicAdd(&p.counters[bgq], 1);
    is_last = (old == nsplit - 1);
    if (is_last) p.counters[bgq] = 0;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // ---- combine the splits of (b, g, q-group) in split order ------------------
  // (max, sum) of every (split, row) go to shared memory (the K/V buffers are
  // free now); each row's split weights are formed there; then thread c owns
  // output column c of every row and accumulates the splits in order, with
  // the loads of all rows of one split in flight together.
  const float* base = p.part + (int64_t)bgq * p.nsplit_max * 64 * DP;
  float* ml = reinterpret_cast<float*>(smem + 64 * DH * 2);        // [nsplit][64][2]
  float* inv = ml + 2 * 64 * AT_MAX_SPLITS;                         // [64]
  for (int e = tid; e < nsplit * 64; e += AT_THREADS) {
    const int s2 = e >> 6, r = e & 63;
    const float* pr = base + ((int64_t)s2 * 64 + r) * DP;
    ml[2 * e] = r < qrows ? __ldcg(&pr[0]) : 0.f;
    ml[2 * e + 1] = r < qrows ? __ldcg(&pr[1]) : 0.f;
  }
  __syncthreads();
  if (tid < 64) {
    float M = -INFINITY;
    for (int s2 = 0; s2 < nsplit; ++s2) M = fmaxf(M, ml[2 * (s2 * 64 + tid)]);
    float lt = 0.f;
    for (int s2 = 0; s2 < nsplit; ++s2) {
      const float ms = ml[2 * (s2 * 64 + tid)];
      const float w = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
      lt += ml[2 * (s2 * 64 + tid) + 1] * w;
      ml[2 * (s2 * 64 + tid)] = w;
    }
    inv[tid] = 1.0f / lt;
  }
  __syncthreads();
  // each warp owns 16 query rows; its lanes cover one row's DH columns with
  // one float4 each (a coalesced 512-byte row read); 8 rows x 2 splits of
  // loads are in flight together and the splits are added in order
  static_assert(DH == 128, "combine maps 32 lanes x float4 onto a 128-wide row");
  for (int rc = warp * 16; rc < warp * 16 + 16 && rc < qrows; rc += 8) {
    float4 o[8];
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) o[rr] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < nsplit; s0 += 2) {
      float4 v[2][8];
      float w[2][8];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int s2 = min(s0 + u, nsplit - 1);
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          const int r = min(rc + rr, qrows - 1);
          v[u][rr] = __ldcg((const float4*)(base + ((int64_t)s2 * 64 + r) * DP + 4) + lane);
          w[u][rr] = (s0 + u < nsplit) ? ml[2 * (s2 * 64 + r)] : 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          o[rr].x += v[u][rr].x * w[u][rr];
          o[rr].y += v[u][rr].y * w[u][rr];
          o[rr].z += v[u][rr].z * w[u][rr];
          o[rr].w += v[u][rr].w * w[u][rr];
        }
    }
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) {
      const int r = rc + rr;
      if (r >= qrows) break;
      const int qr = q0 + r, hh = qr / p.B, i = qr - hh * p.B;
      bf16* dst = p.o + (int64_t)(b * p.B + i) * (p.H * DH) + (int64_t)(g * p.rep + hh) * DH + 4 * lane;
      const float iv = inv[r];
      __nv_bfloat162 t0 = __floats2bfloat162_rn(o[rr].x * iv, o[rr].y * iv);
      __nv_bfloat162 t1 = __floats2bfloat162_rn(o[rr].z * iv, o[rr].w * iv);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&t0);
      pk.y = *reinterpret_cast<uint32_t*>(&t1);
      *reinterpret_cast<uint2*>(dst) = pk;
    }
  }
}

// Splits per (b, g, q-group): about two CTAs per SM over the whole batch.
static int attn_nsplit_target(const dflash_handle* h, int batch, int B) {
  const dflash_config& c = h->cfg;
  const int rep = c.n_heads / c.n_kv_heads, qgroups = (B * rep + 63) / 64;
  const int64_t units = (int64_t)batch * c.n_kv_heads * qgroups;
  return (int)std::min<int64_t>(AT_MAX_SPLITS,
                                std::max<int64_t>(1, (2 * h->num_sms + units - 1) / units));
}

// Keys per split: the longest sequence divided over at most the target split
// count, using splits of at least AT_MIN_SPLIT keys (fewer, longer splits for
// short contexts), rounded up to a multiple of 64.  Splits start at fixed key
// positions, so a key's split does not depend on the other sequences.
int attn_split_keys(const dflash_handle* h, int batch, int B, int cap) {
  const int64_t keys = (int64_t)cap + B;
  int64_t t = attn_nsplit_target(h, batch, B);
  t = std::max<int64_t>(1, std::min<int64_t>(t, (keys + AT_MIN_SPLIT - 1) / AT_MIN_SPLIT));
  int64_t s = (keys + t - 1) / t;
  return (int)(((s + 63) / 64) * 64);
}

size_t attn_scratch_bytes(const dflash_handle* h, int batch, int B) {
  const dflash_config& c = h->cfg;
  const int rep = c.n_heads / c.n_kv_heads, qgroups = (B * rep + 63) / 64;
  return (size_t)batch * c.n_kv_heads * qgroups * attn_nsplit_target(h, batch, B) * 64 *
             (c.head_dim + 4) * sizeof(float) + 256;
}

bool attn_fast_ok(const dflash_handle* h, int B) {
  const dflash_config& c = h->cfg;
  return c.dtype == DFLASH_BF16 && c.head_dim == 128 && h->num_sms > 0 && B >= 1;
}

int attention_fast(dflash_handle* h, cudaStream_t s, const void* q, const void* kc, const void* vc,
                   int cap, const int32_t* len, const void* kb, const void* vb, int batch, int B,
                   void* o, float* scratch) {
  const dflash_config& c = h->cfg;
  constexpr int DH = 128;
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
  p.H = c.n_heads;
  p.G = c.n_kv_heads;
  p.rep = c.n_heads / c.n_kv_heads;
  p.split = attn_split_keys(h, batch, B, cap);
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)DH);
  p.part = scratch;
  p.qgroups = (B * p.rep + 63) / 64;
  p.nsplit_max = (cap + B + p.split - 1) / p.split;
  p.counters = h->d_counters;
  p.status = h->d_status;
  if ((int64_t)batch * p.G * p.qgroups > kMaxTiles) return DFLASH_ERR_SHAPE;
  // main loop: Q + AT_STAGES x (K, V) sub-chunks; combine: Q region + (max,
  // sum) per (split, row) + 64 inverse sums
  const size_t smem = std::max<size_t>((size_t)(64 + 2 * AT_STAGES * AT_KSUB) * DH * 2,
                                       (size_t)64 * DH * 2 + (2 * 64 * AT_MAX_SPLITS + 64) * 4) +
                      128;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attn_split_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return DFLASH_ERR_CUDA;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nsplit_max, p.G, batch * p.qgroups);
  cfg.blockDim = dim3(AT_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  Timer t;
  launch_begin(h, DFLASH_K_ATTENTION, s, &t);
  cudaLaunchKernelEx(&cfg, attn_split_kernel<DH>, p);
  return launch_end(h, s, &t);
}

}  // namespace dflash
