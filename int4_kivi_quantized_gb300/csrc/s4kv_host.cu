// Host side of the s4kv C ABI: argument checks, pool layout, launches and the
// status word. Declarations and the byte format are in include/s4kv.h.

#include "s4kv_common.cuh"

#include <cmath>
#include <cstring>
#include <new>

using namespace s4kv;

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launches go to the current device: it must be the one the cache's pool lives on.
bool on_cache_device(const s4kv_cache* cache) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return dev == cache->device;
}

int check_cfg(const s4kv_config* c) {
  if (!c) return S4KV_ERR_INVALID_ARG;
  if (c->num_layers <= 0 || c->num_pages <= 0 || c->num_kv_heads <= 0 || c->max_slots <= 0)
    return S4KV_ERR_INVALID_ARG;
  // Fail fast on anything but the one supported shape (standard attention with
  // head_dim 128), as the method's product page prescribes.
  if (c->head_dim != kD) return S4KV_ERR_UNSUPPORTED;
  if (c->page_size != kP || c->group_k != kG || c->group_v != kGv) return S4KV_ERR_UNSUPPORTED;
  if (c->dtype != S4KV_F16 && c->dtype != S4KV_BF16) return S4KV_ERR_UNSUPPORTED;
  if (c->bits != 0 && c->bits != 4 && c->bits != 2 && c->bits != 8) return S4KV_ERR_UNSUPPORTED;
  if (c->residual_v < 1 || c->residual_v > 1024) return S4KV_ERR_UNSUPPORTED;
  if (c->num_kv_heads > 64 || c->max_slots > 65536) return S4KV_ERR_UNSUPPORTED;
  if (static_cast<long long>(c->num_pages) * c->num_kv_heads > (1LL << 31) - 1)
    return S4KV_ERR_UNSUPPORTED;
  return S4KV_OK;
}

// Pool: [status 256 B][lens][reserved: one int32 per (slot, kv head)]
// [FP8 only: scales][layer 0][layer 1]...
// Layer: [pages][key rings][value rings], each 256-byte aligned; FP8 pools have
// no rings (every token goes to its page on arrival).
int bits_of(const s4kv_config* c) { return c->bits == 2 ? 2 : c->bits == 8 ? 8 : 4; }

void layout_of(const s4kv_config* c, s4kv_layout* L, size_t* counters_off) {
  const size_t e = 2, H = c->num_kv_heads, S = c->max_slots;
  const int bits = bits_of(c);
  const bool two = bits == 2, fp8 = bits == 8;
  std::memset(L, 0, sizeof(*L));
  L->status_offset = 0;
  L->lens_offset = 256;
  const size_t lens_bytes = static_cast<size_t>(c->num_layers) * S * H * 4;
  const size_t ctr = align_up(L->lens_offset + lens_bytes, 256);
  *counters_off = ctr;
  const size_t ctr_bytes = S * H * 4;
  L->layer_offset = align_up(ctr + ctr_bytes, 256);
  if (fp8) {   // float [num_layers][2][H]: key scales, then value scales
    L->scale_offset = L->layer_offset;
    L->layer_offset = align_up(L->scale_offset + static_cast<size_t>(c->num_layers) * 2 * H * 4, 256);
  }
  L->record_bytes = rec_bytes(bits);
  L->page_stride = L->record_bytes * H;
  if (fp8) {
    L->kcode_offset = Rec<8>::kKc;
    L->vcode_offset = Rec<8>::kVc;
    L->kmeta_offset = L->vmeta_offset = Rec<8>::kBytes;   // no metadata
  } else {
    L->kcode_offset = two ? Rec<2>::kKc : Rec<4>::kKc;
    L->kmeta_offset = two ? Rec<2>::kKm : Rec<4>::kKm;
    L->vcode_offset = two ? Rec<2>::kVc : Rec<4>::kVc;
    L->vmeta_offset = two ? Rec<2>::kVm : Rec<4>::kVm;
  }
  const size_t pages = L->page_stride * static_cast<size_t>(c->num_pages);
  L->kring_row_stride = kD * e;
  L->kring_head_stride = fp8 ? 0 : kG * L->kring_row_stride;
  L->kring_slot_stride = H * L->kring_head_stride;
  L->kring_offset = align_up(pages, 256);
  L->vring_row_stride = kD * e;
  L->vring_head_stride = fp8 ? 0 : static_cast<size_t>(c->residual_v) * L->vring_row_stride;
  L->vring_slot_stride = H * L->vring_head_stride;
  L->vring_offset = align_up(L->kring_offset + S * L->kring_slot_stride, 256);
  L->layer_stride = align_up(L->vring_offset + S * L->vring_slot_stride, 256);
  L->pool_bytes = L->layer_offset + static_cast<size_t>(c->num_layers) * L->layer_stride;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The layer's FP8 scales (key [H], then value [H]); null for KIVI pools.
float* fp8_scales_of(const s4kv_cache* c, int layer) {
  if (c->bits != 8) return nullptr;
  return reinterpret_cast<float*>(c->pool + c->lay.scale_offset) + static_cast<size_t>(layer) * 2 * c->cfg.num_kv_heads;
}

// Scratch of the decode kernel: two (m, l, o) partials per worker warp.
size_t decode_ws_bytes(const s4kv_cache* c, int B, int g, int* grid) {
  const int per_sm = decode_ctas_per_sm(c->decode_impl, B);
  if (grid) *grid = c->num_sms * per_sm;
  const size_t warps = static_cast<size_t>(c->num_sms) * per_sm * decode_warps_per_cta(c->decode_impl);
  return 2 * warps * decode_partial_bytes(g) + decode_meta_bytes(B, c->cfg.num_kv_heads) + warps * decode_trace_bytes_per_warp();
}

}  // namespace

namespace s4kv {
size_t mq_timeline_bytes_per_warp();   // 0 unless built with -DS4KV_DECODE_TRACE
}  // namespace s4kv

extern "C" {

const char* s4kv_strerror(int status) {
  switch (status) {
    case S4KV_OK: return "ok";
    case S4KV_ERR_INVALID_ARG: return "invalid argument";
    case S4KV_ERR_UNSUPPORTED: return "unsupported configuration (head_dim 128, page 16, G 32, Gv 32, fp16/bf16, GQA group <= 8)";
    case S4KV_ERR_CUDA: return "CUDA runtime error";
    case S4KV_ERR_POOL_TOO_SMALL: return "pool smaller than s4kv_cache_bytes()";
    case S4KV_ERR_DEVICE: return "a kernel found invalid caller data (see the status detail)";
    case S4KV_ERR_DEVICE_TIMEOUT: return "a bounded device wait ran out";
    case S4KV_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than s4kv_decode_workspace_bytes()";
    default: return "unknown status";
  }
}

int s4kv_cache_bytes(const s4kv_config* cfg, size_t* pool_bytes, size_t* bytes_per_token_head) {
  const int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!pool_bytes) return S4KV_ERR_INVALID_ARG;
  s4kv_layout L;
  size_t ctr;
  layout_of(cfg, &L, &ctr);
  *pool_bytes = L.pool_bytes;
  if (bytes_per_token_head) *bytes_per_token_head = rec_bytes(bits_of(cfg)) / kP;
  return S4KV_OK;
}

int s4kv_capacity_tokens(const s4kv_config* cfg, double budget_bytes, long long* tokens, long long* pages) {
  if (!cfg || !tokens || !pages || !(budget_bytes >= 0.0)) return S4KV_ERR_INVALID_ARG;
  s4kv_config c = *cfg;
  c.num_pages = 1;
  const int rc = check_cfg(&c);
  if (rc) return rc;
  auto pool_of = [&](long long n) {
    c.num_pages = static_cast<int>(n);
    s4kv_layout L;
    size_t ctr;
    layout_of(&c, &L, &ctr);
    return static_cast<double>(L.pool_bytes);
  };
  // the largest n with pool(n) <= budget; pool grows with n, and n * H_kv < 2^31
  long long lo = 0, hi = ((1LL << 31) - 1) / cfg->num_kv_heads;
  if (hi > 0x7fffffffLL) hi = 0x7fffffffLL;
  if (pool_of(1) > budget_bytes) hi = 0;
  while (lo < hi) {
    const long long mid = lo + (hi - lo + 1) / 2;
    if (pool_of(mid) <= budget_bytes) lo = mid; else hi = mid - 1;
  }
  *pages = lo;
  *tokens = lo * kP;
  return S4KV_OK;
}

int s4kv_kv_bytes(const s4kv_config* cfg, double batch, double tokens, s4kv_kv_bytes_report* out) {
  const int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!out || batch < 0 || tokens < 0) return S4KV_ERR_INVALID_ARG;
  const double L = cfg->num_layers, H = cfg->num_kv_heads, d = cfg->head_dim;
  const double lbh = L * batch * H;
  out->fp16_equiv_bytes = 2.0 * L * batch * tokens * H * d * 2.0;
  out->code_bytes = 2.0 * L * batch * tokens * H * d * (bits_of(cfg) / 8.0);
  if (bits_of(cfg) == 8) {   // FP8: every token in its page, no group metadata, no rings
    out->meta_bytes = 0.0;
    out->residual_bytes = 0.0;
    out->paged_bytes = lbh * std::ceil(tokens / cfg->page_size) * rec_bytes(8);
    return S4KV_OK;
  }
  const double kgroups = std::floor(tokens / cfg->group_k);
  const double vtok = std::fmax(0.0, tokens - cfg->residual_v);
  out->meta_bytes = lbh * (kgroups * d * 8.0 + vtok * (d / cfg->group_v) * 8.0);
  out->residual_bytes = lbh * (cfg->group_k + cfg->residual_v) * d * 2.0;
  out->paged_bytes = lbh * std::ceil(tokens / cfg->page_size) * rec_bytes(bits_of(cfg));
  return S4KV_OK;
}

int s4kv_cache_create(const s4kv_config* cfg, void* d_pool, size_t pool_bytes, s4kv_cache** out) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!d_pool || !out || (reinterpret_cast<uintptr_t>(d_pool) & 255u)) return S4KV_ERR_INVALID_ARG;
  s4kv_cache* c = new (std::nothrow) s4kv_cache;
  if (!c) return S4KV_ERR_INVALID_ARG;
  std::memset(c, 0, sizeof(*c));
  c->cfg = *cfg;
  layout_of(cfg, &c->lay, &c->counters_offset);
  if (pool_bytes < c->lay.pool_bytes) {
    delete c;
    return S4KV_ERR_POOL_TOO_SMALL;
  }
  c->pool = static_cast<char*>(d_pool);
  c->pool_bytes = pool_bytes;
  c->elem_bytes = 2;
  c->wait_ns = 1000000000LL;
  c->tail_cost = 3;
  c->key_split = 1;   // the default: within the tolerance on wide-scale (outlier) key channels
  c->bits = bits_of(cfg);
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess ||
      cudaMemset(c->pool, 0, c->lay.layer_offset) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    delete c;
    return S4KV_ERR_CUDA;
  }
  if (c->bits == 8) {   // every FP8 scale starts at 1.0
    const size_t n = static_cast<size_t>(cfg->num_layers) * 2 * cfg->num_kv_heads;
    float* ones = new (std::nothrow) float[n];
    if (!ones) {
      delete c;
      return S4KV_ERR_INVALID_ARG;
    }
    for (size_t i = 0; i < n; ++i) ones[i] = 1.0f;
    const cudaError_t e = cudaMemcpy(c->pool + c->lay.scale_offset, ones, n * sizeof(float), cudaMemcpyHostToDevice);
    delete[] ones;
    if (e != cudaSuccess) {
      delete c;
      return S4KV_ERR_CUDA;
    }
  }
  *out = c;
  return S4KV_OK;
}

int s4kv_set_fp8_scales(s4kv_cache* cache, int layer, const float* k_scale, const float* v_scale, void* stream) {
  if (!cache || layer < 0 || layer >= cache->cfg.num_layers || !k_scale || !v_scale) return S4KV_ERR_INVALID_ARG;
  if (cache->bits != 8) return S4KV_ERR_UNSUPPORTED;
  const int H = cache->cfg.num_kv_heads;
  float buf[2 * 64];
  for (int h = 0; h < H; ++h) {
    if (!(k_scale[h] > 0.0f) || !(v_scale[h] > 0.0f) || std::isinf(k_scale[h]) || std::isinf(v_scale[h]))
      return S4KV_ERR_INVALID_ARG;
    buf[h] = k_scale[h];
    buf[H + h] = v_scale[h];
  }
  // work already queued on `stream` keeps the old scales
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return S4KV_ERR_CUDA;
  char* dst = cache->pool + cache->lay.scale_offset + static_cast<size_t>(layer) * 2 * H * sizeof(float);
  return cudaMemcpy(dst, buf, 2 * H * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess ? S4KV_OK : S4KV_ERR_CUDA;
}

int s4kv_cache_destroy(s4kv_cache* cache) {
  if (!cache) return S4KV_ERR_INVALID_ARG;
  delete cache;
  return S4KV_OK;
}

int s4kv_get_layout(const s4kv_cache* cache, s4kv_layout* out) {
  if (!cache || !out) return S4KV_ERR_INVALID_ARG;
  *out = cache->lay;
  return S4KV_OK;
}

int s4kv_set_option(s4kv_cache* cache, int option, long long value) {
  if (!cache) return S4KV_ERR_INVALID_ARG;
  switch (option) {
    case S4KV_OPT_DECODE_WARPS:
      if (value < 0 || value > (1 << 24)) return S4KV_ERR_INVALID_ARG;
      cache->decode_warps = static_cast<int>(value);
      return S4KV_OK;
    case S4KV_OPT_DECODE_IMPL:
      if (value != 0 && value != 1) return S4KV_ERR_INVALID_ARG;
      cache->decode_impl = static_cast<int>(value);
      return S4KV_OK;
    case S4KV_OPT_TAIL_COST:
      if (value < 1 || value > 1024) return S4KV_ERR_INVALID_ARG;
      cache->tail_cost = static_cast<int>(value);
      return S4KV_OK;
    case S4KV_OPT_MQ_KERNEL:
      if (value < 0 || value > 3) return S4KV_ERR_INVALID_ARG;
      cache->mq_kernel = static_cast<int>(value);
      return S4KV_OK;
    case S4KV_OPT_KEY_SPLIT:
      if (value != 0 && value != 1) return S4KV_ERR_INVALID_ARG;
      cache->key_split = static_cast<int>(value);
      return S4KV_OK;
    case S4KV_OPT_WAIT_NS:
      if (value < 0) return S4KV_ERR_INVALID_ARG;
      cache->wait_ns = value;
      return S4KV_OK;
    default:
      return S4KV_ERR_INVALID_ARG;
  }
}

int s4kv_append(s4kv_cache* cache, int layer, const void* k, const void* v, int num_new_tokens,
                const int32_t* cu_new, const int32_t* slot_ids, const int32_t* seq_lens_before,
                const int32_t* block_table, int bt_stride, int n, void* stream) {
  if (!cache || layer < 0 || layer >= cache->cfg.num_layers || n < 0 || num_new_tokens < 0)
    return S4KV_ERR_INVALID_ARG;
  if (n == 0) return S4KV_OK;
  if (!on_cache_device(cache)) return S4KV_ERR_INVALID_ARG;
  if (n > cache->cfg.max_slots || n > 8192) return S4KV_ERR_INVALID_ARG;
  if (!cu_new || !seq_lens_before || !block_table || bt_stride <= 0) return S4KV_ERR_INVALID_ARG;
  if (num_new_tokens > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return S4KV_ERR_INVALID_ARG;
  const s4kv_config& c = cache->cfg;
  char* base = cache->pool + cache->lay.layer_offset + static_cast<size_t>(layer) * cache->lay.layer_stride;
  AppendArgs a;
  a.pages = base;
  a.kring = base + cache->lay.kring_offset;
  a.vring = base + cache->lay.vring_offset;
  a.lens = reinterpret_cast<int*>(cache->pool + cache->lay.lens_offset) +
           static_cast<size_t>(layer) * c.max_slots * c.num_kv_heads;
  a.status = reinterpret_cast<int*>(cache->pool + cache->lay.status_offset);
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.cu_new = cu_new;
  a.slot_ids = slot_ids;
  a.seq_lens_before = seq_lens_before;
  a.block_table = block_table;
  a.kring_slot = cache->lay.kring_slot_stride / 2;
  a.kring_head = cache->lay.kring_head_stride / 2;
  a.vring_slot = cache->lay.vring_slot_stride / 2;
  a.vring_head = cache->lay.vring_head_stride / 2;
  a.bt_stride = bt_stride;
  a.n = n;
  a.num_new = num_new_tokens;
  a.H = c.num_kv_heads;
  a.R = c.residual_v;
  a.num_pages = c.num_pages;
  a.max_slots = c.max_slots;
  a.dtype = c.dtype;
  a.bits = cache->bits;
  a.fp8_scale = fp8_scales_of(cache, layer);
  const long long bound = static_cast<long long>(c.num_kv_heads) * (3LL * n + num_new_tokens / 32 + 1);
  const long long cap = static_cast<long long>(cache->num_sms) * append_ctas_per_sm();
  const int grid = static_cast<int>(bound < cap ? bound : cap);
  cudaError_t e = launch_append(a, grid, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? S4KV_OK : S4KV_ERR_CUDA;
}

int s4kv_decode_workspace_bytes(const s4kv_cache* cache, int B, int num_q_heads, int max_seq_len,
                                size_t* bytes) {
  if (!cache || !bytes || B < 0 || B > 4096 || num_q_heads <= 0 || max_seq_len < 0)
    return S4KV_ERR_INVALID_ARG;
  if (num_q_heads % cache->cfg.num_kv_heads) return S4KV_ERR_INVALID_ARG;
  const int g = num_q_heads / cache->cfg.num_kv_heads;
  if (g > kMaxGroup) return S4KV_ERR_UNSUPPORTED;
  *bytes = decode_ws_bytes(cache, B, g, nullptr);
  return *bytes ? S4KV_OK : S4KV_ERR_CUDA;
}

namespace {
// Decode kernel variant of the key split: the rest of q' rides in columns 4..7 of
// the same MMA when a kv head serves at most 4 query heads (3), else a second MMA (2).
int split_impl(int g) { return g <= 4 ? 3 : 2; }

// Arguments common to both attention entry points (checked by the callers).
DecodeArgs attention_args(s4kv_cache* cache, int layer, const void* q, int num_q_heads,
                          const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                          const int32_t* slot_ids, int B, float sm_scale, void* out, int out_dtype,
                          void* workspace, int max_seq_len) {
  const s4kv_config& c = cache->cfg;
  char* base = cache->pool + cache->lay.layer_offset + static_cast<size_t>(layer) * cache->lay.layer_stride;
  DecodeArgs a;
  a.pages = base;
  a.kring = base + cache->lay.kring_offset;
  a.vring = base + cache->lay.vring_offset;
  a.lens = reinterpret_cast<const int*>(cache->pool + cache->lay.lens_offset) +
           static_cast<size_t>(layer) * c.max_slots * c.num_kv_heads;
  a.status = reinterpret_cast<int*>(cache->pool + cache->lay.status_offset);
  a.q = static_cast<const uint16_t*>(q);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.slot_ids = slot_ids;
  a.out = out;
  a.ws = static_cast<float*>(workspace);
  a.kring_slot = cache->lay.kring_slot_stride / 2;
  a.kring_head = cache->lay.kring_head_stride / 2;
  a.vring_slot = cache->lay.vring_slot_stride / 2;
  a.vring_head = cache->lay.vring_head_stride / 2;
  a.wait_ns = cache->wait_ns;
  const float scale = sm_scale > 0.0f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(kD));
  a.sm_scale_log2 = scale * 1.4426950408889634f;
  a.bt_stride = bt_stride;
  a.B = B;
  a.Hq = num_q_heads;
  a.H = c.num_kv_heads;
  a.g = num_q_heads / c.num_kv_heads;
  a.R = c.residual_v;
  a.num_pages = c.num_pages;
  a.max_slots = c.max_slots;
  a.dtype = c.dtype;
  a.bits = cache->bits;
  a.fp8_scale = fp8_scales_of(cache, layer);
  a.out_dtype = out_dtype;
  a.max_warps = cache->decode_warps;
  a.tail_cost = cache->tail_cost;
  a.max_seq_len = max_seq_len;
  a.nq = 1;
  a.tw = 1;
  a.pcols = a.g;
  a.key_split = cache->key_split;
  a.mq_kernel = cache->mq_kernel;
  a.knew = nullptr;
  a.vnew = nullptr;
  a.lens_w = nullptr;
  a.gbar = nullptr;
  return a;
}

// Columns a multi-query warp holds (both page formats).
int mq_cols_per_warp(const s4kv_cache*) { return 2 * kMaxGroup; }

// Scratch of the multi-query kernel: two partials of a warp's columns per worker warp.
size_t mq_ws_bytes(const s4kv_cache* c, int B, int* grid) {
  const int per_sm = decode_ctas_per_sm(0, B);
  if (grid) *grid = c->num_sms * per_sm;
  const size_t warps = static_cast<size_t>(c->num_sms) * per_sm * decode_warps_per_cta(0);
  return 2 * warps * decode_partial_bytes(mq_cols_per_warp(c)) + decode_meta_bytes(B, c->cfg.num_kv_heads) +
         warps * (decode_trace_bytes_per_warp() + mq_timeline_bytes_per_warp());
}

// Shape limits of the multi-query path: nq tokens, g heads per kv head. KIVI
// pages need the chunk inside the value window (nq <= R); FP8 pages have none.
int mq_shape_ok(const s4kv_cache* c, int nq, int g) {
  if (nq < 1 || nq > 16) return S4KV_ERR_INVALID_ARG;
  if ((c->bits != 8 && nq > c->cfg.residual_v) || nq * g > 96) return S4KV_ERR_UNSUPPORTED;
  return S4KV_OK;
}
}  // namespace

int s4kv_decode_attention(s4kv_cache* cache, int layer, const void* q, int num_q_heads,
                          const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                          const int32_t* slot_ids, int B, float sm_scale, void* out, int out_dtype,
                          void* workspace, size_t ws_bytes, int max_seq_len, void* stream) {
  if (!cache || layer < 0 || layer >= cache->cfg.num_layers || B < 0 || max_seq_len < 0)
    return S4KV_ERR_INVALID_ARG;
  if (!on_cache_device(cache)) return S4KV_ERR_INVALID_ARG;
  if (B == 0) return S4KV_OK;
  const s4kv_config& c = cache->cfg;
  if (B > 4096 || num_q_heads <= 0 || num_q_heads % c.num_kv_heads) return S4KV_ERR_INVALID_ARG;
  const int g = num_q_heads / c.num_kv_heads;
  if (g > kMaxGroup) return S4KV_ERR_UNSUPPORTED;
  if (!q || !out || !block_table || !seq_lens || bt_stride <= 0 || !aligned16(q) || !aligned16(out))
    return S4KV_ERR_INVALID_ARG;
  if (out_dtype != S4KV_F32 && out_dtype != c.dtype) return S4KV_ERR_INVALID_ARG;
  int grid = 0;
  const size_t need = decode_ws_bytes(cache, B, g, &grid);
  if (grid <= 0) return S4KV_ERR_CUDA;
  if (ws_bytes < need) return S4KV_ERR_WORKSPACE_TOO_SMALL;
  if (!workspace || !aligned16(workspace)) return S4KV_ERR_INVALID_ARG;
  if (cache->bits != 4 && cache->decode_impl == 1) return S4KV_ERR_UNSUPPORTED;   // FFMA path: 4-bit only
  DecodeArgs a = attention_args(cache, layer, q, num_q_heads, block_table, bt_stride, seq_lens, slot_ids, B,
                                sm_scale, out, out_dtype, workspace, max_seq_len);
  a.grid_warps = grid * decode_warps_per_cta(cache->decode_impl);
  // the tensor-core path with the key split is kernel variant 2, or 3 where the GQA
  // group leaves half the MMA's columns free (KIVI codes only: FP8 keys meet the
  // query unscaled, exactly in f16)
  const int impl = cache->decode_impl == 0 && cache->key_split && cache->bits != 8 ? split_impl(g)
                                                                                   : cache->decode_impl;
  cudaError_t e = launch_decode(a, impl, grid, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? S4KV_OK : S4KV_ERR_CUDA;
}

int s4kv_decode_step(s4kv_cache* cache, int layer, const void* k_new, const void* v_new, const void* q,
                     int num_q_heads, const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                     const int32_t* slot_ids, int B, float sm_scale, void* out, int out_dtype, void* workspace,
                     size_t ws_bytes, int max_seq_len, void* stream) {
  if (!cache || layer < 0 || layer >= cache->cfg.num_layers || B < 0 || max_seq_len < 0)
    return S4KV_ERR_INVALID_ARG;
  if (!on_cache_device(cache)) return S4KV_ERR_INVALID_ARG;
  if (B == 0) return S4KV_OK;
  const s4kv_config& c = cache->cfg;
  if (B > 4096 || num_q_heads <= 0 || num_q_heads % c.num_kv_heads) return S4KV_ERR_INVALID_ARG;
  const int g = num_q_heads / c.num_kv_heads;
  if (g > kMaxGroup) return S4KV_ERR_UNSUPPORTED;
  if (!q || !out || !block_table || !seq_lens || bt_stride <= 0 || !aligned16(q) || !aligned16(out))
    return S4KV_ERR_INVALID_ARG;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return S4KV_ERR_INVALID_ARG;
  if (out_dtype != S4KV_F32 && out_dtype != c.dtype) return S4KV_ERR_INVALID_ARG;
  if (cache->decode_impl == 1) return S4KV_ERR_UNSUPPORTED;   // the step runs on the tensor-core paths
  int grid = 0;
  const size_t need = decode_ws_bytes(cache, B, g, &grid);
  if (grid <= 0) return S4KV_ERR_CUDA;
  if (ws_bytes < need) return S4KV_ERR_WORKSPACE_TOO_SMALL;
  if (!workspace || !aligned16(workspace)) return S4KV_ERR_INVALID_ARG;
  DecodeArgs a = attention_args(cache, layer, q, num_q_heads, block_table, bt_stride, seq_lens, slot_ids, B,
                                sm_scale, out, out_dtype, workspace, max_seq_len);
  a.grid_warps = grid * decode_warps_per_cta(0);
  a.knew = static_cast<const uint16_t*>(k_new);
  a.vnew = static_cast<const uint16_t*>(v_new);
  a.lens_w = const_cast<int*>(a.lens);
  a.gbar = reinterpret_cast<unsigned*>(cache->pool + cache->lay.status_offset) + ST_BAR_COUNT;
  const int impl = cache->key_split && cache->bits != 8 ? split_impl(g) : 0;
  cudaError_t e = launch_decode_step(a, impl, grid, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return S4KV_ERR_CUDA;
  }
  return S4KV_OK;
}

int s4kv_multi_query_workspace_bytes(const s4kv_cache* cache, int B, int num_q_tokens, int num_q_heads,
                                     int max_seq_len, size_t* bytes) {
  if (!cache || !bytes || B < 0 || B > 4096 || num_q_heads <= 0 || max_seq_len < 0)
    return S4KV_ERR_INVALID_ARG;
  if (num_q_heads % cache->cfg.num_kv_heads) return S4KV_ERR_INVALID_ARG;
  const int rc = mq_shape_ok(cache, num_q_tokens, num_q_heads / cache->cfg.num_kv_heads);
  if (rc != S4KV_OK) return rc;
  *bytes = mq_ws_bytes(cache, B, nullptr);
  return *bytes ? S4KV_OK : S4KV_ERR_CUDA;
}

int s4kv_multi_query_attention(s4kv_cache* cache, int layer, const void* q, int num_q_tokens, int num_q_heads,
                               const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                               const int32_t* slot_ids, int B, float sm_scale, void* out, int out_dtype,
                               void* workspace, size_t ws_bytes, int max_seq_len, void* stream) {
  if (!cache || layer < 0 || layer >= cache->cfg.num_layers || B < 0 || max_seq_len < 0)
    return S4KV_ERR_INVALID_ARG;
  if (!on_cache_device(cache)) return S4KV_ERR_INVALID_ARG;
  if (B == 0) return S4KV_OK;
  const s4kv_config& c = cache->cfg;
  if (B > 4096 || num_q_heads <= 0 || num_q_heads % c.num_kv_heads) return S4KV_ERR_INVALID_ARG;
  const int g = num_q_heads / c.num_kv_heads;
  const int rc = mq_shape_ok(cache, num_q_tokens, g);
  if (rc != S4KV_OK) return rc;
  if (!q || !out || !block_table || !seq_lens || bt_stride <= 0 || !aligned16(q) || !aligned16(out))
    return S4KV_ERR_INVALID_ARG;
  if (out_dtype != S4KV_F32 && out_dtype != c.dtype) return S4KV_ERR_INVALID_ARG;
  int grid = 0;
  const size_t need = mq_ws_bytes(cache, B, &grid);
  if (grid <= 0) return S4KV_ERR_CUDA;
  if (ws_bytes < need) return S4KV_ERR_WORKSPACE_TOO_SMALL;
  if (!workspace || !aligned16(workspace)) return S4KV_ERR_INVALID_ARG;
  DecodeArgs a = attention_args(cache, layer, q, num_q_heads, block_table, bt_stride, seq_lens, slot_ids, B,
                                sm_scale, out, out_dtype, workspace, max_seq_len);
  a.grid_warps = grid * decode_warps_per_cta(0);
  a.nq = num_q_tokens;
  a.pcols = mq_cols_per_warp(cache);
  a.tw = (num_q_tokens * g + a.pcols - 1) / a.pcols;
  cudaError_t e = launch_mq(a, grid, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? S4KV_OK : S4KV_ERR_CUDA;
}

int s4kv_dequant_debug(s4kv_cache* cache, int layer, int slot, const int32_t* block_table_row,
                       int seq_len, float* out_k, float* out_v, void* stream) {
  if (!cache || layer < 0 || layer >= cache->cfg.num_layers || slot < 0 ||
      slot >= cache->cfg.max_slots || seq_len < 0)
    return S4KV_ERR_INVALID_ARG;
  if (seq_len == 0) return S4KV_OK;
  if (!block_table_row || !out_k || !out_v) return S4KV_ERR_INVALID_ARG;
  if (!on_cache_device(cache)) return S4KV_ERR_INVALID_ARG;
  const s4kv_config& c = cache->cfg;
  char* base = cache->pool + cache->lay.layer_offset + static_cast<size_t>(layer) * cache->lay.layer_stride;
  DequantArgs a;
  a.pages = base;
  a.kring = base + cache->lay.kring_offset;
  a.vring = base + cache->lay.vring_offset;
  a.lens = reinterpret_cast<const int*>(cache->pool + cache->lay.lens_offset) +
           static_cast<size_t>(layer) * c.max_slots * c.num_kv_heads;
  a.status = reinterpret_cast<int*>(cache->pool + cache->lay.status_offset);
  a.bt_row = block_table_row;
  a.out_k = out_k;
  a.out_v = out_v;
  a.kring_slot = cache->lay.kring_slot_stride / 2;
  a.kring_head = cache->lay.kring_head_stride / 2;
  a.vring_slot = cache->lay.vring_slot_stride / 2;
  a.vring_head = cache->lay.vring_head_stride / 2;
  a.slot = slot;
  a.T = seq_len;
  a.H = c.num_kv_heads;
  a.R = c.residual_v;
  a.num_pages = c.num_pages;
  a.max_slots = c.max_slots;
  a.dtype = c.dtype;
  a.bits = cache->bits;
  a.fp8_scale = fp8_scales_of(cache, layer);
  cudaError_t e = launch_dequant(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? S4KV_OK : S4KV_ERR_CUDA;
}

int s4kv_get_status(s4kv_cache* cache, void* stream, int* detail) {
  if (!cache) return S4KV_ERR_INVALID_ARG;
  int words[3] = {0, 0, 0};
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return S4KV_ERR_CUDA;
  int* st = reinterpret_cast<int*>(cache->pool + cache->lay.status_offset);
  if (cudaMemcpy(words, st, sizeof(words), cudaMemcpyDeviceToHost) != cudaSuccess) return S4KV_ERR_CUDA;
  if (detail) *detail = words[1];
  if (words[0] != 0) {
    if (cudaMemset(st, 0, sizeof(words)) != cudaSuccess) return S4KV_ERR_CUDA;
    // a barrier that ran out of time may have left its arrival count behind
    if (words[0] == S4KV_ERR_DEVICE_TIMEOUT && cudaMemset(st + ST_BAR_COUNT, 0, 2 * sizeof(int)) != cudaSuccess)
      return S4KV_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return S4KV_ERR_CUDA;
    return words[0];
  }
  return S4KV_OK;
}

}  // extern "C"
