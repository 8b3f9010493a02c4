// Host-side common entry points: status strings, configuration checks,
// weight shapes, device properties and the programmatic-dependent-launch switch.
#include <atomic>
#include <mutex>

#include "ft_internal.cuh"

namespace ft_host {

static std::atomic<int> g_pdl{1};
static std::mutex g_sm_mu;
static int g_sm_count[64] = {0};

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64) {
    std::lock_guard<std::mutex> lk(g_sm_mu);
    if (g_sm_count[dev] > 0) return g_sm_count[dev];
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) {
    std::lock_guard<std::mutex> lk(g_sm_mu);
    g_sm_count[dev] = n;
  }
  return n;
}

bool pdl_enabled() { return g_pdl.load() != 0; }

int smem_per_sm() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess) return 0;
  return n;
}

static bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int check_cfg(const ft_block_cfg* c) {
  if (!c) return FT_ERR_INVALID_ARG;
  if (c->hidden <= 0 || c->n_q <= 0 || c->n_kv <= 0 || c->head_dim <= 0 || c->inter <= 0)
    return FT_ERR_INVALID_ARG;
  if (c->n_q % c->n_kv) return FT_ERR_INVALID_ARG;
  if (!(c->rms_eps >= 0.0f) || !(c->rope_base > 0.0f)) return FT_ERR_INVALID_ARG;
  if (c->w_group != 128) return FT_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return FT_ERR_UNSUPPORTED;
  if (!pow2(c->had_block) || c->head_dim % c->had_block) return FT_ERR_INVALID_ARG;
  if (c->kv_group != c->head_dim) return FT_ERR_UNSUPPORTED;
  if (c->n_q / c->n_kv > 8) return FT_ERR_UNSUPPORTED;
  if (c->hidden % 128 || c->inter % 128) return FT_ERR_UNSUPPORTED;
  if ((c->n_q * c->head_dim) % 128) return FT_ERR_UNSUPPORTED;
  if (((c->n_q + 2 * c->n_kv) * c->head_dim) % 128) return FT_ERR_UNSUPPORTED;
  if (c->weight_format != FT_WFMT_INT4 && c->weight_format != FT_WFMT_E4M3) return FT_ERR_INVALID_ARG;
  return FT_OK;
}

}  // namespace ft_host

extern "C" {

const char* ft_status_string(int s) {
  switch (s) {
    case FT_OK: return "ok";
    case FT_ERR_INVALID_ARG: return "invalid argument (NULL or misaligned pointer, bad size, overlap)";
    case FT_ERR_UNSUPPORTED: return "unsupported shape or option";
    case FT_ERR_WORKSPACE: return "workspace or packed buffer too small";
    case FT_ERR_CAPACITY: return "batch exceeds cache capacity";
    case FT_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

int ft_validate_cfg(const ft_block_cfg* cfg) { return ft_host::check_cfg(cfg); }

int ft_weight_shape(const ft_block_cfg* c, int role, int32_t* n_out, int32_t* k_in) {
  int st = ft_host::check_cfg(c);
  if (st != FT_OK) return st;
  if (!n_out || !k_in) return FT_ERR_INVALID_ARG;
  switch (role) {
    case FT_W_QKV: *n_out = (c->n_q + 2 * c->n_kv) * c->head_dim; *k_in = c->hidden; break;
    case FT_W_O: *n_out = c->hidden; *k_in = c->n_q * c->head_dim; break;
    case FT_W_GATEUP: *n_out = 2 * c->inter; *k_in = c->hidden; break;
    case FT_W_DOWN: *n_out = c->hidden; *k_in = c->inter; break;
    default: return FT_ERR_INVALID_ARG;
  }
  return FT_OK;
}

size_t ft_packed_weight_bytes(const ft_block_cfg* c, int role) {
  int32_t n, k;
  if (ft_weight_shape(c, role, &n, &k) != FT_OK) return 0;
  return (size_t)(n / ft::kRowTile) * (size_t)(k / ft::kWGroup) * (size_t)ft::slab_bytes_of(c->weight_format);
}

int ft_set_pdl(int enabled) { return ft_host::g_pdl.exchange(enabled ? 1 : 0); }

}  // extern "C"
