// LM-head argmax without caller-provided workspace.
//
// Some callers cannot hand the library a workspace: a serving loop whose
// device memory is fully reserved up front by its own pool, or a
// latency-critical path that must not call cudaMalloc (which can synchronise
// the device and has no latency bound).  For them this entry point keeps its
// scratch in one file-scope device array of fixed size.  Every GPU that loads
// the library reserves that array until the process exits.
#include <mutex>

#include "common.cuh"

namespace dflash {

// Limits of the static scratch.
constexpr int NA_MAX_ROWS = 16;          // rows per call
constexpr int NA_MAX_HIDDEN = 8192;      // hidden size D
constexpr int NA_MAX_VOCAB = 262144;     // vocabulary V
constexpr int NA_MAX_CTAS = 320;         // streaming CTAs per launch (SMs x CTAs per SM)

constexpr size_t NA_HF_BYTES = (size_t)NA_MAX_ROWS * NA_MAX_HIDDEN * 2;              // bf16 rows
constexpr size_t NA_PART_BYTES = (size_t)2 * NA_MAX_CTAS * 16 * 128 * sizeof(float);  // k-split partials
constexpr size_t NA_AMX_BYTES = (size_t)(NA_MAX_VOCAB / 128) * NA_MAX_ROWS * 16;     // top-2 records
constexpr size_t NA_BYTES = NA_HF_BYTES + NA_PART_BYTES + NA_AMX_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NA_BYTES];

// Device address of the array, looked up once per device (host code cannot
// use the symbol itself: on the host it names a stand-in, not device memory).
static std::mutex g_na_mu;
static void* g_na_ptr[64] = {nullptr};

static int noalloc_scratch(int dev, void** out) {
  if (dev < 0 || dev >= 64) return DFLASH_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_na_mu);
  if (!g_na_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DFLASH_ERR_CUDA;
    g_na_ptr[dev] = p;
  }
  *out = g_na_ptr[dev];
  return DFLASH_OK;
}

}  // namespace dflash

using namespace dflash;

extern "C" int dflash_lm_head_argmax_noalloc(dflash_handle* h, const float* x, int32_t rows,
                                              const float* norm_gain, int32_t* ids,
                                              float* top2_gap, dflash_stream_t st) {
  if (!h || !x || !norm_gain || !ids || rows < 0) return DFLASH_ERR_INVALID_ARG;
  if (rows == 0) return DFLASH_OK;
  const dflash_config& c = h->cfg;
  if (!h->have_maps) return DFLASH_ERR_UNSUPPORTED;       // bf16 streaming handles only
  if (rows > NA_MAX_ROWS || c.hidden > NA_MAX_HIDDEN || c.vocab > NA_MAX_VOCAB ||
      wstream_scratch_bytes(h, rows) > NA_PART_BYTES)
    return DFLASH_ERR_STATIC_LIMIT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DFLASH_ERR_CUDA;
  void* base = nullptr;
  int rc = noalloc_scratch(dev, &base);
  if (rc) return rc;
  char* p = (char*)base;
  void* hf = p;
  float* partial = (float*)(p + NA_HF_BYTES);
  float4* amx = (float4*)(p + NA_HF_BYTES + NA_PART_BYTES);
  cudaStream_t s = (cudaStream_t)st;
  // final RMSNorm into bf16 rows, then the streamed LM head with its argmax
  // epilogue (the tile counters live in the handle and return to zero by
  // themselves; the rest of the scratch is fully written before it is read)
  rc = rmsnorm_rows(h, s, DFLASH_F32, DFLASH_BF16, x, c.hidden, hf, c.hidden, norm_gain, rows,
                    c.hidden, c.rms_eps, 0);
  if (rc) return rc;
  WLaunch L;
  L.nmap = 1;
  L.wmaps[0] = &h->map_lm;
  L.nseg = 1;
  WSeg g{};
  g.t0 = 0;
  g.t1 = (c.vocab + 127) / 128;
  g.kind = SK_ARGMAX;
  g.map = 0;
  g.n_valid = c.vocab;
  L.seg[0] = g;
  L.nsrc = 1;
  L.a_src[0] = hf;
  L.a_ld = c.hidden;
  L.K = c.hidden;
  L.M = rows;
  L.ids = ids;
  L.gap = top2_gap;
  L.rps_out = 0;
  L.anchor = nullptr;
  return wstream(h, s, DFLASH_K_LM_HEAD, L, partial, amx);
}
