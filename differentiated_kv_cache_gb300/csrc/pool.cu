// pool.cu — host implementation of the libdkv C ABI (include/dkv.h).
//
// The pool owns every device structure of DiffKV's memory manager (unified
// pages, circular free page list, bidirectional page tables, counters) plus
// the kernels' scratch. Calls queue kernels on the caller's stream and never
// synchronise; request-state checks use a host mirror of the request table,
// which dkv_pool_clear_error re-reads from the device.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>

#include "dkv_kernels.cuh"

using namespace dkv;

struct dkv_pool {
  Pool P;
};

namespace {

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

int round16(int x) { return (x + 15) & ~15; }

// Unified page layout of one tier for t tokens; returns bytes used.
int layout_tier(int t, int kbits, int vbits, TierGeom* tg) {
  const int g = 8 / vbits;
  const int sizes[6] = {t * kD * kbits / 8, (t / g) * 128, 4 * t, 4 * t, 4 * t, 4 * t};
  int o = 0;
  for (int s = 0; s < 6; s++) {
    tg->off[s] = o;
    o = round16(o + sizes[s]);
  }
  tg->t = t;
  tg->kbytes = kD * kbits / 8;
  tg->magic = (uint32_t)((1ull << 32) / (unsigned)t + 1);
  return tg->off[5] + sizes[5];
}

// Tokens per page: the override, or the largest multiple of g that fits.
int fit_tier(int page_bytes, int kbits, int vbits, int override_t, TierGeom* tg) {
  const int g = 8 / vbits;
  if (override_t) {
    if (override_t < g || override_t % g) return -1;
    return layout_tier(override_t, kbits, vbits, tg) <= page_bytes ? override_t : -1;
  }
  int best = -1;
  for (int t = g; t * 32 <= page_bytes * 8; t += g) {
    TierGeom tmp;
    if (layout_tier(t, kbits, vbits, &tmp) <= page_bytes) best = t; else break;
  }
  if (best > 0) layout_tier(best, kbits, vbits, tg);
  return best;
}

template <typename T>
cudaError_t dev_alloc(Pool& P, T** ptr, size_t count) {
  void* p = nullptr;
  const size_t bytes = std::max<size_t>(count * sizeof(T), 256);
  cudaError_t e = cudaMalloc(&p, bytes);
  if (e != cudaSuccess) return e;
  P.allocations.push_back(p);
  *ptr = reinterpret_cast<T*>(p);
  return cudaSuccess;
}

void free_all(Pool& P) {
  for (void* p : P.allocations) cudaFree(p);
  P.allocations.clear();
}

__global__ void k_init_list(int* list, int n) {
  for (int x = blockIdx.x * blockDim.x + threadIdx.x; x < n; x += gridDim.x * blockDim.x) list[x] = x;
}

int validate(const dkv_config* c) {
  if (!c) return DKV_ERR_ARG;
  if (c->n_layers < 1 || c->n_kv_heads < 1 || c->n_pages < 1 || c->max_requests < 1 || c->max_seq_len < 1)
    return DKV_ERR_ARG;
  if (c->page_bytes < 64 || c->page_bytes % 16) return DKV_ERR_ARG;
  if (c->recent_window < 0 || c->prompt_grant_slack < 0) return DKV_ERR_ARG;
  if (std::isnan(c->alpha_h) || std::isnan(c->alpha_l)) return DKV_ERR_ARG;
  if (c->mid_enabled && (!c->lo_enabled || std::isnan(c->alpha_m))) return DKV_ERR_ARG;
  if (c->head_dim != kD || c->group_size < 1 || c->group_size > kMaxG || c->obs_window != kObs)
    return DKV_ERR_UNSUPPORTED;
  return DKV_OK;
}

int cuda_err(cudaError_t e) { return e == cudaSuccess ? DKV_OK : DKV_ERR_CUDA; }

// Device buffers are read and written with 16-byte vector accesses.
bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" {

const char* dkv_strerror(int code) {
  switch (code) {
    case DKV_OK: return "ok";
    case DKV_ERR_ARG: return "invalid argument";
    case DKV_ERR_CUDA: return "CUDA runtime error";
    case DKV_ERR_STATE: return "request slot in the wrong state";
    case DKV_ERR_NO_PAGES: return "free page list exhausted";
    case DKV_ERR_TABLE_FULL: return "page table row or grant full";
    case DKV_ERR_TIMEOUT: return "bounded device wait expired";
    case DKV_ERR_CHECK: return "device consistency check failed";
    case DKV_ERR_UNSUPPORTED: return "configuration not supported by the kernels";
    case DKV_ERR_SCRATCH: return "call needs more than the fixed scratch array holds";
    default: return "unknown error";
  }
}

int dkv_pool_create(const dkv_config* cfg, int cuda_device, dkv_pool** out) {
  if (!out) return DKV_ERR_ARG;
  *out = nullptr;
  int rc = validate(cfg);
  if (rc) return rc;
  TierGeom hi{}, lo{}, mid{};
  if (fit_tier(cfg->page_bytes, 8, 4, cfg->tokens_per_hi_page, &hi) < 0) return DKV_ERR_ARG;
  if (fit_tier(cfg->page_bytes, 4, 2, cfg->tokens_per_lo_page, &lo) < 0) return DKV_ERR_ARG;
  const bool three = cfg->mid_enabled != 0;
  if (three) {
    if (fit_tier(cfg->page_bytes, 8, 2, cfg->tokens_per_mid_page, &mid) < 0) return DKV_ERR_ARG;
    // the three-tier path runs the page-per-copy attention kernel only
    if (hi.t % kChunk || lo.t % kChunk || mid.t % kChunk) return DKV_ERR_UNSUPPORTED;
  }
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || cuda_device < 0 || cuda_device >= ndev) return DKV_ERR_ARG;
  DeviceGuard guard(cuda_device);
  dkv_pool* pool = new (std::nothrow) dkv_pool();
  if (!pool) return DKV_ERR_CUDA;
  Pool& P = pool->P;
  P.cfg = *cfg;
  P.device = cuda_device;
  if (cudaDeviceGetAttribute(&P.sm_count, cudaDevAttrMultiProcessorCount, cuda_device) != cudaSuccess) {
    delete pool;
    return DKV_ERR_CUDA;
  }
  PoolView& v = P.pv;
  v.n_pages = cfg->n_pages;
  v.page_bytes = cfg->page_bytes;
  v.n_layers = cfg->n_layers;
  v.hkv = cfg->n_kv_heads;
  v.G = cfg->group_size;
  v.max_req = cfg->max_requests;
  v.max_seq = cfg->max_seq_len;
  v.L = (cfg->max_seq_len + hi.t - 1) / hi.t + 1;
  v.lo_enabled = cfg->lo_enabled ? 1 : 0;
  v.window = cfg->recent_window;
  v.slack = cfg->prompt_grant_slack;
  v.reclaim = cfg->reclaim_in_decode ? 1 : 0;
  v.hi = hi;
  v.lo = lo;
  v.mid = mid;
  v.mid_enabled = three ? 1 : 0;
  v.Lm = three ? (cfg->max_seq_len + mid.t - 1) / mid.t + 1 : 0;
  v.Lrow = v.L + v.Lm;
  v.cstride = three ? 8 : 4;
  Scratch& s = P.sc;
  const size_t heads = (size_t)cfg->n_layers * cfg->max_requests * cfg->n_kv_heads;
  const size_t units = (size_t)cfg->max_requests * cfg->n_kv_heads;
  const size_t max_tokens = (size_t)cfg->max_requests * cfg->max_seq_len;
  const int G = cfg->group_size;
  s.nkb_cap = (cfg->max_seq_len + kKeyBlock - 1) / kKeyBlock;
  s.grant_cap = (cfg->max_seq_len + hi.t - 1) / hi.t + cfg->prompt_grant_slack;
  // chunks of a head: its tiers' token counts rounded up to 16 each
  s.max_chunks = (cfg->max_seq_len + kChunk - 1) / kChunk + (three ? 2 : 1);
  s.max_splits = s.max_chunks / 8 + 2;   // attention partials per head (>= 8 chunks per warp)
  s.max_scan = (cfg->max_seq_len + 1 + 2047) / 2048;   // generation-phase scan CTAs per head
  // victim-key partials per head: a warp of every attention epilogue block
  // of the head (>= 64 chunks a block)
  v.max_vp = (s.max_chunks + 63) / 64 * kVictimWarps;
  cudaError_t e = cudaSuccess;
  auto A = [&](auto** ptr, size_t n) {
    if (e == cudaSuccess) e = dev_alloc(P, ptr, n);
  };
  A(&v.pages, (size_t)cfg->n_pages * cfg->page_bytes);
  A(&v.list, (size_t)cfg->n_pages);
  A(&v.table, heads * v.Lrow);
  A(&v.counts, heads * v.cstride);
  A(&v.req, (size_t)cfg->n_layers * cfg->max_requests * 4);
  A(&v.ctl, 1);
  A(&v.call, 1);
  A(&v.vparts, heads * v.max_vp);
  A(&v.vstamp, heads);
  A(&v.alpha, (size_t)cfg->n_layers * cfg->n_kv_heads);
  A(&v.alpha_m, (size_t)cfg->n_layers * cfg->n_kv_heads);
  A(&s.partial, units * s.nkb_cap * kObs * G);
  A(&s.lse2, units * kObs * G);
  A(&s.score, max_tokens * cfg->n_kv_heads);
  A(&s.tokinfo, max_tokens * cfg->n_kv_heads);
  A(&s.bcnt, units * s.nkb_cap);
  A(&s.bbase, units * s.nkb_cap);
  A(&s.bcnt_m, units * s.nkb_cap);
  A(&s.bbase_m, units * s.nkb_cap);
  A(&s.unit_mid, units);
  A(&s.rank2pos, units * (three ? 3 : 2) * cfg->max_seq_len);
  A(&s.unit_info, units);
  A(&s.grant_ids, units * s.grant_cap);
  A(&s.pbase, 4);
  A(&s.dplan, units);
  A(&s.dscan, units * s.max_scan);
  A(&s.darrive, units);
  A(&s.apart, units * s.max_splits * (G * kD + 2 * kMaxG));
  A(&s.alogit, units * s.max_chunks * G * kChunk);
  A(&s.alse, units * G);
  if (e == cudaSuccess) e = cudaMemset(s.darrive, 0, units * sizeof(int));
  // stamps -1: no head has victim keys yet
  if (e == cudaSuccess) e = cudaMemset(v.vparts, 0xff, heads * v.max_vp * sizeof(VictimPart));
  if (e == cudaSuccess) e = cudaMemset(v.vstamp, 0xff, heads * sizeof(int4));
  if (e == cudaSuccess) e = cudaMemset(v.pages, 0, (size_t)cfg->n_pages * cfg->page_bytes);
  if (e == cudaSuccess) e = cudaMemset(v.table, 0xff, heads * v.Lrow * sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(v.counts, 0, heads * v.cstride * sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(v.req, 0, (size_t)cfg->n_layers * cfg->max_requests * 4 * sizeof(int));
  if (e == cudaSuccess) {
    Ctl c{};
    c.start = 0;
    c.end = (unsigned long long)cfg->n_pages;
    c.error_info = -1;
    e = cudaMemcpy(v.ctl, &c, sizeof(Ctl), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) {        // every head starts with the configuration's pair
    std::vector<float2> al((size_t)cfg->n_layers * cfg->n_kv_heads, make_float2(cfg->alpha_h, cfg->alpha_l));
    e = cudaMemcpy(v.alpha, al.data(), al.size() * sizeof(float2), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) {
    std::vector<float> am((size_t)cfg->n_layers * cfg->n_kv_heads, three ? cfg->alpha_m : 0.0f);
    e = cudaMemcpy(v.alpha_m, am.data(), am.size() * sizeof(float), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) {
    k_init_list<<<256, 256>>>(v.list, cfg->n_pages);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = configure_kernels();
  // the allocation-free attention's array on this device, in this context
  if (e == cudaSuccess) e = static_scratch_address(&P.static_base);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    free_all(P);
    delete pool;
    return DKV_ERR_CUDA;
  }
  P.h_active.assign((size_t)cfg->n_layers * cfg->max_requests, 0);
  P.h_n0.assign(P.h_active.size(), 0);
  P.h_n.assign(P.h_active.size(), 0);
  *out = pool;
  return DKV_OK;
}

int dkv_pool_destroy(dkv_pool* pool) {
  if (!pool) return DKV_OK;
  DeviceGuard guard(pool->P.device);
  const cudaError_t e = cudaDeviceSynchronize();
  free_all(pool->P);
  delete pool;
  return cuda_err(e);
}

int dkv_pool_geometry(const dkv_pool* pool, dkv_geometry* out) {
  if (!pool || !out) return DKV_ERR_ARG;
  const PoolView& v = pool->P.pv;
  out->t_hi = v.hi.t;
  out->t_lo = v.lo.t;
  out->table_len = v.L;
  for (int s = 0; s < 6; s++) {
    out->hi_off[s] = v.hi.off[s];
    out->lo_off[s] = v.lo.off[s];
  }
  TierGeom tmp;
  out->hi_used = layout_tier(v.hi.t, 8, 4, &tmp);
  out->lo_used = layout_tier(v.lo.t, 4, 2, &tmp);
  out->t_mid = v.mid_enabled ? v.mid.t : 0;
  out->mid_table_len = v.Lm;
  out->row_len = v.Lrow;
  out->count_stride = v.cstride;
  for (int s = 0; s < 6; s++) out->mid_off[s] = v.mid_enabled ? v.mid.off[s] : 0;
  out->mid_used = v.mid_enabled ? layout_tier(v.mid.t, 8, 2, &tmp) : 0;
  return DKV_OK;
}

int dkv_compact_step(dkv_pool* pool, int32_t layer, int32_t mode, int32_t n_req, const int32_t* req_slots,
                     const int32_t* seq_lens, const void* k, const void* v, const void* q_obs,
                     const float* scores_in, float* scores_out, void* stream) {
  if (!pool || !req_slots || !k || !v) return DKV_ERR_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(q_obs) || !aligned4(scores_in) || !aligned4(scores_out))
    return DKV_ERR_ARG;
  Pool& P = pool->P;
  const dkv_config& c = P.cfg;
  if (layer < 0 || layer >= c.n_layers || n_req < 1 || n_req > c.max_requests || n_req > kMaxCallReq)
    return DKV_ERR_ARG;
  if (mode != DKV_PROMPT && mode != DKV_DECODE) return DKV_ERR_ARG;
  for (int i = 0; i < n_req; i++) {
    if (req_slots[i] < 0 || req_slots[i] >= c.max_requests) return DKV_ERR_ARG;
    for (int j = 0; j < i; j++)
      if (req_slots[j] == req_slots[i]) return DKV_ERR_ARG;
  }
  const size_t base = (size_t)layer * c.max_requests;
  CallArgs args;
  args.n_req = n_req;
  args.pad = 0;
  if (mode == DKV_PROMPT) {
    if (!seq_lens || (!q_obs && !scores_in)) return DKV_ERR_ARG;
    long long tok = 0;
    for (int i = 0; i < n_req; i++) {
      if (seq_lens[i] < 1 || seq_lens[i] > c.max_seq_len) return DKV_ERR_ARG;
      if (P.h_active[base + req_slots[i]]) return DKV_ERR_STATE;
      args.slots[i] = req_slots[i];
      args.lens[i] = seq_lens[i];
      args.tok0[i] = tok;
      tok += seq_lens[i];
    }
    args.tok0[n_req] = tok;
  } else {
    if (seq_lens || q_obs || scores_in || scores_out) return DKV_ERR_ARG;
    if (c.recent_window < 1) return DKV_ERR_ARG;
    SlotArgs sa;
    sa.n = n_req;
    for (int i = 0; i < n_req; i++) {
      if (!P.h_active[base + req_slots[i]]) return DKV_ERR_STATE;
      if (P.h_n[base + req_slots[i]] + 1 > c.max_seq_len) return DKV_ERR_ARG;
      sa.slots[i] = req_slots[i];
    }
    DeviceGuard guard(P.device);
    const cudaError_t e = launch_decode(P, layer, sa, static_cast<const __half*>(k), static_cast<const __half*>(v),
                                        reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return DKV_ERR_CUDA;
    for (int i = 0; i < n_req; i++) P.h_n[base + req_slots[i]] += 1;
    return DKV_OK;
  }
  DeviceGuard guard(P.device);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_setup(P, args, st);
  if (e != cudaSuccess) return DKV_ERR_CUDA;
  int max_len = 0;
  for (int i = 0; i < n_req; i++) max_len = std::max(max_len, seq_lens[i]);
  e = launch_prompt(P, layer, n_req, max_len, args.tok0[n_req], static_cast<const __half*>(k),
                    static_cast<const __half*>(v),
                    static_cast<const __half*>(q_obs), nullptr, scores_in, scores_out, st);
  if (e != cudaSuccess) return DKV_ERR_CUDA;
  for (int i = 0; i < n_req; i++) {
    P.h_active[base + req_slots[i]] = 1;
    P.h_n0[base + req_slots[i]] = seq_lens[i];
    P.h_n[base + req_slots[i]] = seq_lens[i];
  }
  return DKV_OK;
}

int dkv_prefill_attention(dkv_pool* pool, int32_t n_req, const int32_t* seq_lens, const void* q, const void* k,
                          const void* v, float* out, float* lse_obs, void* stream) {
  if (!pool || !seq_lens || !q || !k || !v || !out) return DKV_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned4(lse_obs)) return DKV_ERR_ARG;
  Pool& P = pool->P;
  const dkv_config& c = P.cfg;
  if (n_req < 1 || n_req > kMaxCallReq) return DKV_ERR_ARG;
  CallArgs args;
  args.n_req = n_req;
  args.pad = 0;
  long long tok = 0;
  int max_len = 0;
  for (int i = 0; i < n_req; i++) {
    if (seq_lens[i] < 1 || seq_lens[i] > c.max_seq_len) return DKV_ERR_ARG;
    args.slots[i] = -1;
    args.lens[i] = seq_lens[i];
    args.tok0[i] = tok;
    tok += seq_lens[i];
    max_len = std::max(max_len, seq_lens[i]);
  }
  args.tok0[n_req] = tok;
  DeviceGuard guard(P.device);
  const cudaError_t e = launch_prefill(P, args, max_len, static_cast<const __half*>(q), static_cast<const __half*>(k),
                                       static_cast<const __half*>(v), out, lse_obs,
                                       reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DKV_OK : DKV_ERR_CUDA;
}

int dkv_compact_step_prefilled(dkv_pool* pool, int32_t layer, int32_t n_req, const int32_t* req_slots,
                               const int32_t* seq_lens, const void* k, const void* v, const void* q_obs,
                               const float* lse_obs, float* scores_out, void* stream) {
  if (!pool || !req_slots || !seq_lens || !k || !v || !q_obs || !lse_obs) return DKV_ERR_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(q_obs) || !aligned4(lse_obs) || !aligned4(scores_out))
    return DKV_ERR_ARG;
  Pool& P = pool->P;
  const dkv_config& c = P.cfg;
  if (layer < 0 || layer >= c.n_layers || n_req < 1 || n_req > c.max_requests || n_req > kMaxCallReq)
    return DKV_ERR_ARG;
  const size_t base = (size_t)layer * c.max_requests;
  CallArgs args;
  args.n_req = n_req;
  args.pad = 0;
  long long tok = 0;
  int max_len = 0;
  for (int i = 0; i < n_req; i++) {
    if (req_slots[i] < 0 || req_slots[i] >= c.max_requests) return DKV_ERR_ARG;
    for (int j = 0; j < i; j++)
      if (req_slots[j] == req_slots[i]) return DKV_ERR_ARG;
    if (seq_lens[i] < 1 || seq_lens[i] > c.max_seq_len) return DKV_ERR_ARG;
  }
  for (int i = 0; i < n_req; i++) {
    if (P.h_active[base + req_slots[i]]) return DKV_ERR_STATE;
    args.slots[i] = req_slots[i];
    args.lens[i] = seq_lens[i];
    args.tok0[i] = tok;
    tok += seq_lens[i];
    max_len = std::max(max_len, seq_lens[i]);
  }
  args.tok0[n_req] = tok;
  DeviceGuard guard(P.device);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_setup(P, args, st);
  if (e != cudaSuccess) return DKV_ERR_CUDA;
  e = launch_prompt(P, layer, n_req, max_len, tok, static_cast<const __half*>(k), static_cast<const __half*>(v),
                    static_cast<const __half*>(q_obs), lse_obs, nullptr, scores_out, st);
  if (e != cudaSuccess) return DKV_ERR_CUDA;
  for (int i = 0; i < n_req; i++) {
    P.h_active[base + req_slots[i]] = 1;
    P.h_n0[base + req_slots[i]] = seq_lens[i];
    P.h_n[base + req_slots[i]] = seq_lens[i];
  }
  return DKV_OK;
}

int dkv_decode_attention(dkv_pool* pool, int32_t layer, int32_t n_req, const int32_t* req_slots, const void* q,
                         float* out, int32_t update_scores, void* stream) {
  if (!pool || !req_slots || !q || !out) return DKV_ERR_ARG;
  if (!aligned16(q) || !aligned16(out)) return DKV_ERR_ARG;
  Pool& P = pool->P;
  const dkv_config& c = P.cfg;
  if (layer < 0 || layer >= c.n_layers || n_req < 1 || n_req > c.max_requests || n_req > kMaxCallReq)
    return DKV_ERR_ARG;
  const size_t base = (size_t)layer * c.max_requests;
  SlotArgs sa;
  sa.n = n_req;
  int max_tokens = 1;
  for (int i = 0; i < n_req; i++) {
    if (req_slots[i] < 0 || req_slots[i] >= c.max_requests) return DKV_ERR_ARG;
    for (int j = 0; j < i; j++)
      if (req_slots[j] == req_slots[i]) return DKV_ERR_ARG;
    if (!P.h_active[base + req_slots[i]]) return DKV_ERR_STATE;
    sa.slots[i] = req_slots[i];
    max_tokens = std::max(max_tokens, P.h_n[base + req_slots[i]]);
  }
  DeviceGuard guard(P.device);
  const cudaError_t e = launch_attention(P, layer, sa, max_tokens, static_cast<const __half*>(q), out,
                                         update_scores ? 1 : 0, reinterpret_cast<cudaStream_t>(stream));
  return cuda_err(e);
}

// Same checks and kernels as dkv_decode_attention; scratch in the static
// array of attention.cu (for callers that cannot allocate device memory).
int dkv_decode_attention_static(dkv_pool* pool, int32_t layer, int32_t n_req, const int32_t* req_slots,
                                const void* q, float* out, int32_t update_scores, void* stream) {
  if (!pool || !req_slots || !q || !out) return DKV_ERR_ARG;
  if (!aligned16(q) || !aligned16(out)) return DKV_ERR_ARG;
  Pool& P = pool->P;
  const dkv_config& c = P.cfg;
  if (layer < 0 || layer >= c.n_layers || n_req < 1 || n_req > c.max_requests || n_req > kMaxCallReq)
    return DKV_ERR_ARG;
  const size_t base = (size_t)layer * c.max_requests;
  SlotArgs sa;
  sa.n = n_req;
  int max_tokens = 1;
  for (int i = 0; i < n_req; i++) {
    if (req_slots[i] < 0 || req_slots[i] >= c.max_requests) return DKV_ERR_ARG;
    for (int j = 0; j < i; j++)
      if (req_slots[j] == req_slots[i]) return DKV_ERR_ARG;
    if (!P.h_active[base + req_slots[i]]) return DKV_ERR_STATE;
    sa.slots[i] = req_slots[i];
    max_tokens = std::max(max_tokens, P.h_n[base + req_slots[i]]);
  }
  const int update = update_scores ? 1 : 0;
  if (attention_static_bytes(P, n_req * c.n_kv_heads, max_tokens, update) > DKV_ATTN_STATIC_SCRATCH_BYTES)
    return DKV_ERR_SCRATCH;
  DeviceGuard guard(P.device);
  const cudaError_t e = launch_attention_static(P, layer, sa, max_tokens, static_cast<const __half*>(q), out,
                                                update, reinterpret_cast<cudaStream_t>(stream));
  return cuda_err(e);
}

int dkv_pool_set_thresholds(dkv_pool* pool, int32_t layer, const float* alpha_h, const float* alpha_l,
                            void* stream) {
  if (!pool || !alpha_h || !alpha_l) return DKV_ERR_ARG;
  Pool& P = pool->P;
  const dkv_config& c = P.cfg;
  if (layer < 0 || layer >= c.n_layers) return DKV_ERR_ARG;
  std::vector<float2> al(c.n_kv_heads);
  for (int h = 0; h < c.n_kv_heads; h++) {
    if (std::isnan(alpha_h[h]) || std::isnan(alpha_l[h])) return DKV_ERR_ARG;
    al[h] = make_float2(alpha_h[h], alpha_l[h]);
  }
  DeviceGuard guard(P.device);
  // from pageable memory: the call returns once the values are staged
  const cudaError_t e = cudaMemcpyAsync(P.pv.alpha + (size_t)layer * c.n_kv_heads, al.data(),
                                        al.size() * sizeof(float2), cudaMemcpyHostToDevice,
                                        reinterpret_cast<cudaStream_t>(stream));
  return cuda_err(e);
}

int dkv_pool_set_mid_thresholds(dkv_pool* pool, int32_t layer, const float* alpha_m, void* stream) {
  if (!pool || !alpha_m) return DKV_ERR_ARG;
  Pool& P = pool->P;
  const dkv_config& c = P.cfg;
  if (layer < 0 || layer >= c.n_layers || !P.pv.mid_enabled) return DKV_ERR_ARG;
  std::vector<float> am(c.n_kv_heads);
  for (int h = 0; h < c.n_kv_heads; h++) {
    if (std::isnan(alpha_m[h])) return DKV_ERR_ARG;
    am[h] = alpha_m[h];
  }
  DeviceGuard guard(P.device);
  const cudaError_t e = cudaMemcpyAsync(P.pv.alpha_m + (size_t)layer * c.n_kv_heads, am.data(),
                                        am.size() * sizeof(float), cudaMemcpyHostToDevice,
                                        reinterpret_cast<cudaStream_t>(stream));
  return cuda_err(e);
}

int dkv_free_request(dkv_pool* pool, int32_t req_slot, void* stream) {
  if (!pool) return DKV_ERR_ARG;
  Pool& P = pool->P;
  const dkv_config& c = P.cfg;
  if (req_slot < 0 || req_slot >= c.max_requests) return DKV_ERR_ARG;
  bool any = false;
  for (int l = 0; l < c.n_layers; l++) any |= P.h_active[(size_t)l * c.max_requests + req_slot] != 0;
  if (!any) return DKV_ERR_STATE;
  DeviceGuard guard(P.device);
  const cudaError_t e = launch_free(P, req_slot, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return DKV_ERR_CUDA;
  for (int l = 0; l < c.n_layers; l++) {
    const size_t x = (size_t)l * c.max_requests + req_slot;
    P.h_active[x] = 0;
    P.h_n0[x] = 0;
    P.h_n[x] = 0;
  }
  return DKV_OK;
}

int dkv_pool_status(dkv_pool* pool, dkv_status* out) {
  if (!pool || !out) return DKV_ERR_ARG;
  Pool& P = pool->P;
  DeviceGuard guard(P.device);
  if (cudaDeviceSynchronize() != cudaSuccess) return DKV_ERR_CUDA;
  Ctl c;
  if (cudaMemcpy(&c, P.pv.ctl, sizeof(Ctl), cudaMemcpyDeviceToHost) != cudaSuccess) return DKV_ERR_CUDA;
  const size_t heads = (size_t)P.cfg.n_layers * P.cfg.max_requests * P.cfg.n_kv_heads;
  const int cs = P.pv.cstride;
  std::vector<int> cnt(heads * cs);
  if (cudaMemcpy(cnt.data(), P.pv.counts, cnt.size() * sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DKV_ERR_CUDA;
  out->error = c.error;
  out->error_info = c.error ? c.error_info : -1;
  out->list_start = (int64_t)c.start;
  out->list_end = (int64_t)c.end;
  out->free_pages = (int64_t)(c.end - c.start);
  out->hi_tokens = out->lo_tokens = out->hi_pages = out->lo_pages = out->mid_tokens = out->mid_pages = 0;
  for (size_t h = 0; h < heads; h++) {
    out->hi_tokens += cnt[cs * h];
    out->lo_tokens += cnt[cs * h + 1];
    out->hi_pages += cnt[cs * h + 2];
    out->lo_pages += cnt[cs * h + 3];
    if (cs > 4) {
      out->mid_tokens += cnt[cs * h + 4];
      out->mid_pages += cnt[cs * h + 5];
    }
  }
  return DKV_OK;
}

int dkv_pool_clear_error(dkv_pool* pool) {
  if (!pool) return DKV_ERR_ARG;
  Pool& P = pool->P;
  DeviceGuard guard(P.device);
  if (cudaDeviceSynchronize() != cudaSuccess) return DKV_ERR_CUDA;
  Ctl c;
  if (cudaMemcpy(&c, P.pv.ctl, sizeof(Ctl), cudaMemcpyDeviceToHost) != cudaSuccess) return DKV_ERR_CUDA;
  c.error = 0;
  c.error_info = -1;
  if (cudaMemcpy(P.pv.ctl, &c, sizeof(Ctl), cudaMemcpyHostToDevice) != cudaSuccess) return DKV_ERR_CUDA;
  // a step cut short can leave generation-phase scan arrivals behind, and an
  // attention call cut short a head's stamps beside partials it did not
  // finish: the next generation steps scan
  if (cudaMemset(P.sc.darrive, 0, (size_t)P.cfg.max_requests * P.cfg.n_kv_heads * sizeof(int)) != cudaSuccess)
    return DKV_ERR_CUDA;
  if (cudaMemset(P.pv.vstamp, 0xff,
                 (size_t)P.cfg.n_layers * P.cfg.max_requests * P.cfg.n_kv_heads * sizeof(int4)) != cudaSuccess)
    return DKV_ERR_CUDA;
  std::vector<int> rq((size_t)P.cfg.n_layers * P.cfg.max_requests * 4);
  if (cudaMemcpy(rq.data(), P.pv.req, rq.size() * sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DKV_ERR_CUDA;
  for (size_t x = 0; x < P.h_active.size(); x++) {
    P.h_active[x] = rq[4 * x];
    P.h_n0[x] = rq[4 * x + 1];
    P.h_n[x] = rq[4 * x + 2];
  }
  return DKV_OK;
}

int dkv_pool_export(dkv_pool* pool, dkv_snapshot* out) {
  if (!pool || !out) return DKV_ERR_ARG;
  Pool& P = pool->P;
  const dkv_config& c = P.cfg;
  DeviceGuard guard(P.device);
  if (cudaDeviceSynchronize() != cudaSuccess) return DKV_ERR_CUDA;
  const size_t heads = (size_t)c.n_layers * c.max_requests * c.n_kv_heads;
  cudaError_t e = cudaSuccess;
  auto cp = [&](void* dst, const void* src, size_t bytes) {
    if (dst && e == cudaSuccess) e = cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost);
  };
  cp(out->pages, P.pv.pages, (size_t)c.n_pages * c.page_bytes);
  cp(out->free_list, P.pv.list, (size_t)c.n_pages * sizeof(int));
  cp(out->table, P.pv.table, heads * P.pv.Lrow * sizeof(int));
  cp(out->head_counts, P.pv.counts, heads * P.pv.cstride * sizeof(int));
  cp(out->req_state, P.pv.req, (size_t)c.n_layers * c.max_requests * 4 * sizeof(int));
  if (out->pointers && e == cudaSuccess) {
    Ctl ctl;
    e = cudaMemcpy(&ctl, P.pv.ctl, sizeof(Ctl), cudaMemcpyDeviceToHost);
    out->pointers[0] = (int64_t)ctl.start;
    out->pointers[1] = (int64_t)ctl.end;
  }
  return cuda_err(e);
}

}  // extern "C"
