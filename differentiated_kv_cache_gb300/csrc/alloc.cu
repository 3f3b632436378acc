// alloc.cu — the coordination phase of parallel KV compaction (DiffKV,
// memory management): page grants and reclaims by exclusive prefix sums over
// all heads of a call against the circular free page list, and the updates of
// the bidirectional page table. Each kernel here is one CTA of 1024 threads;
// per-head work is spread over the threads and joined by block-wide scans.
#include "dkv_kernels.cuh"

namespace dkv {

constexpr int kCoordThreads = 1024;

// Copy the call's host arrays into the pool's device CallArgs.
__global__ void k_setup(PoolView pv, CallArgs args) {
  pdl_launch_dependents();        // the call's first kernel may launch; it waits for this one
  CallArgs* c = pv.call;
  const int n = args.n_req;
  for (int x = threadIdx.x; x < n; x += blockDim.x) {
    c->slots[x] = args.slots[x];
    c->lens[x] = args.lens[x];
    c->tok0[x] = args.tok0[x];
  }
  if (threadIdx.x == 0) {
    c->n_req = n;
    c->tok0[n] = args.tok0[n];
  }
}

// Exclusive scan of one int per thread over the whole block; returns the
// thread's exclusive prefix and writes the block total to *total.
__device__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int s = 1; s < 32; s <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, s);
    if (lane >= s) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, s);
      if (lane >= s) w += y;
    }
    if (lane < nw) s_warp[lane] = w;
  }
  __syncthreads();
  const int excl = x - v + (warp > 0 ? s_warp[warp - 1] : 0);
  const int tot = s_warp[nw - 1];
  __syncthreads();
  *total = tot;
  return excl;
}

// In-place exclusive scan of arr[0..n) in shared memory over the whole block
// (each thread scans a contiguous run); returns the total.
__device__ int block_scan_array(int* arr, int n, int* s_warp) {
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int a0 = min(n, (int)threadIdx.x * per), a1 = min(n, a0 + per);
  int sum = 0;
  for (int x = a0; x < a1; x++) sum += arr[x];
  int total;
  int run = block_exclusive_scan(sum, s_warp, &total);
  for (int x = a0; x < a1; x++) {
    const int v = arr[x];
    arr[x] = run;
    run += v;
  }
  __syncthreads();
  return total;
}

__device__ __forceinline__ void latch_error(PoolView& pv, int code, int info) {
  if (atomicCAS(&pv.ctl->error, 0, code) == 0) pv.ctl->error_info = info;
}

// ---------------------------------------------------------------------------
// Prompt coordination (Figure 6): per head an all-hi grant of
// ceil(N0/T_hi)+slack pages taken at the list start by one prefix sum; hi
// pages from the left of the grant, lo pages from the right; the unused
// middle pages appended at the list end by a second prefix sum; table rows,
// counters and request state written. Three launches over all heads: (1) per
// head tier counts, key-block bases and page needs; (2) grant offsets (every
// CTA scans the per-head grants of the call), the list check and the reads
// of the granted page IDs; (3) reclaim offsets, reclaim writes, table rows
// and counters. Every check precedes every write of the pool's state: (1)
// and (2) write only scratch, and a failed check latches the sticky status
// that turns the later launches into no-ops. All grant reads (2) complete
// before any reclaim write (3), which may reuse list entries once the list
// wraps.
// ---------------------------------------------------------------------------
constexpr int kPlanWarps = 8;   // heads per CTA in the prompt coordination

__global__ void __launch_bounds__(32 * kPlanWarps) k_prompt_plan_heads(PoolView pv, Scratch sc) {
  if (!dependent_begin(pv)) return;
  const CallArgs* ca = pv.call;
  const int n_units = ca->n_req * pv.hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x * kPlanWarps + warp;
  if (u >= n_units) return;
  const int n0 = ca->lens[u / pv.hkv];
  const int nkb = (n0 + kKeyBlock - 1) / kKeyBlock;
  int a = 0, b = 0, m = 0;
  for (int k0 = 0; k0 < nkb; k0 += 32) {
    const int kb = k0 + lane;
    const size_t bx = (size_t)u * sc.nkb_cap + kb;
    const int2 c = kb < nkb ? sc.bcnt[bx] : make_int2(0, 0);
    const int cm = pv.mid_enabled && kb < nkb ? sc.bcnt_m[bx] : 0;
    int x = c.x, y = c.y, z = cm;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const int xo = __shfl_up_sync(0xffffffffu, x, s), yo = __shfl_up_sync(0xffffffffu, y, s);
      const int zo = __shfl_up_sync(0xffffffffu, z, s);
      if (lane >= s) { x += xo; y += yo; z += zo; }
    }
    if (kb < nkb) {
      sc.bbase[bx] = make_int2(a + x - c.x, b + y - c.y);
      if (pv.mid_enabled) sc.bbase_m[bx] = m + z - cm;
    }
    a += __shfl_sync(0xffffffffu, x, 31);
    b += __shfl_sync(0xffffffffu, y, 31);
    m += __shfl_sync(0xffffffffu, z, 31);
  }
  if (lane == 0) {
    const int gh = (n0 + pv.hi.t - 1) / pv.hi.t + pv.slack;
    const int nhp = (a + pv.hi.t - 1) / pv.hi.t, nlp = (b + pv.lo.t - 1) / pv.lo.t;
    const int nmp = pv.mid_enabled ? (m + pv.mid.t - 1) / pv.mid.t : 0;
    if (nhp + nmp + nlp > gh || nhp + nlp > pv.L || nmp > pv.Lm) latch_error(pv, DKV_ERR_TABLE_FULL, u);
    sc.unit_info[u] = make_int4(gh, a, b, max(0, gh - nhp - nmp - nlp));
    if (pv.mid_enabled) sc.unit_mid[u] = m;
  }
}

__global__ void __launch_bounds__(32 * kPlanWarps) k_prompt_plan_grant(PoolView pv, Scratch sc) {
  if (!dependent_begin(pv)) return;          // a head's pages do not fit its grant or row
  extern __shared__ int s_g[];    // [unit] grant pages -> exclusive offsets
  __shared__ int s_warp[32];
  const CallArgs* ca = pv.call;
  const int n_units = ca->n_req * pv.hkv;
  for (int x = threadIdx.x; x < n_units; x += blockDim.x) s_g[x] = sc.unit_info[x].x;
  __syncthreads();
  const int tot_g = block_scan_array(s_g, n_units, s_warp);
  const unsigned long long start = pv.ctl->start, end = pv.ctl->end;
  if ((unsigned long long)tot_g > end - start) {   // every CTA sees the same
    if (blockIdx.x == 0 && threadIdx.x == 0) latch_error(pv, DKV_ERR_NO_PAGES, -1);
    return;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    sc.pbase[0] = start;
    sc.pbase[1] = end;
    sc.pbase[2] = (unsigned long long)tot_g;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x * kPlanWarps + warp;
  if (u >= n_units) return;
  const int gh = sc.unit_info[u].x;
  int* gid = sc.grant_ids + (size_t)u * sc.grant_cap;
  for (int x = lane; x < gh; x += 32) gid[x] = pv.list[(start + (unsigned long long)(s_g[u] + x)) % pv.n_pages];
}

__global__ void __launch_bounds__(32 * kPlanWarps) k_prompt_plan_commit(PoolView pv, int layer, Scratch sc) {
  if (!dependent_begin(pv)) return;
  extern __shared__ int s_r[];    // [unit] reclaimed pages -> exclusive offsets
  __shared__ int s_warp[32];
  const CallArgs* ca = pv.call;
  const int n_units = ca->n_req * pv.hkv;
  for (int x = threadIdx.x; x < n_units; x += blockDim.x) s_r[x] = sc.unit_info[x].w;
  __syncthreads();
  const int tot_r = block_scan_array(s_r, n_units, s_warp);
  const unsigned long long start = sc.pbase[0], end = sc.pbase[1], tot_g = sc.pbase[2];
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    pv.ctl->start = start + tot_g;
    pv.ctl->end = end + (unsigned long long)tot_r;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x * kPlanWarps + warp;
  if (u >= n_units) return;
  const int i = u / pv.hkv, kvh = u % pv.hkv, slot = ca->slots[i];
  const int4 ui = sc.unit_info[u];
  const int gh = ui.x, nhp = (ui.y + pv.hi.t - 1) / pv.hi.t, nlp = (ui.z + pv.lo.t - 1) / pv.lo.t;
  const int nm = pv.mid_enabled ? sc.unit_mid[u] : 0;
  const int nmp = pv.mid_enabled ? (nm + pv.mid.t - 1) / pv.mid.t : 0;   // grant pages nhp .. nhp+nmp-1
  const int* gid = sc.grant_ids + (size_t)u * sc.grant_cap;
  for (int x = nhp + nmp + lane; x < gh - nlp; x += 32)
    pv.list[(end + (unsigned long long)(s_r[u] + x - nhp - nmp)) % pv.n_pages] = gid[x];
  int* row = pv.row(layer, slot, kvh);
  for (int e = lane; e < pv.Lrow; e += 32) {
    int v = -1;
    if (e < nhp) v = gid[e];
    else if (e < pv.L && e >= pv.L - nlp) v = gid[gh - 1 - (pv.L - 1 - e)];
    else if (e >= pv.L && e < pv.L + nmp) v = gid[nhp + e - pv.L];   // the one-way mid part
    row[e] = v;
  }
  if (lane == 0) {
    int* cn = pv.cnt(layer, slot, kvh);
    cn[0] = ui.y; cn[1] = ui.z; cn[2] = nhp; cn[3] = nlp;
    if (pv.mid_enabled) { cn[4] = nm; cn[5] = nmp; }
    if (kvh == 0) {
      int* rq = pv.rq(layer, slot);
      rq[0] = 1; rq[1] = ca->lens[i]; rq[2] = ca->lens[i]; rq[3] = 0;
    }
  }
}

// ---------------------------------------------------------------------------
// Generation-phase coordination: new pages for every head that needs one, by
// one prefix sum at the list start (per head hi, lo, then mid); emptied tail pages
// (reclaim_in_decode) by one prefix sum at the list end; table rows,
// counters and the request lengths updated. All checks precede every write.
// ---------------------------------------------------------------------------
// MID: a three-tier pool (the two-tier instance compiles the mid tier out)
template <bool MID>
__global__ void __launch_bounds__(kCoordThreads) k_decode_alloc(PoolView pv, int layer, Scratch sc,
                                                                 SlotArgs sa) {
  pdl_launch_dependents();        // k_decode_apply may launch; it waits for this grid
  if (pv.noop()) return;
  extern __shared__ int s_list[];  // [k n_units] the list entries from the start: the pages a grant can take
  __shared__ int s_warp[32];
  __shared__ int s_err, s_info;
  const int n_units = sa.n * pv.hkv;
  const int per = (n_units + blockDim.x - 1) / blockDim.x;
  const int u0 = threadIdx.x * per, u1 = min(n_units, u0 + per);
  if (threadIdx.x == 0) { s_err = 0; s_info = -1; }
  // The list counters and the entries from the start (a head takes at most a
  // page of each tier): only this kernel moves or reads them during a
  // generation step, so they load while the plans finish.
  const unsigned long long start = pv.ctl->start, end = pv.ctl->end;
  constexpr int per_head = MID ? 3 : 2;
  for (int x = threadIdx.x; x < per_head * n_units; x += blockDim.x)
    s_list[x] = pv.list[(start + (unsigned long long)x) % pv.n_pages];
  pdl_wait();                     // the plans of k_decode_plan
  if (pv.noop_after_wait()) return;
  __syncthreads();
  int my_a = 0, my_f = 0;
  for (int u = u0; u < u1; u++) {
    const DecodePlan& p = sc.dplan[u];
    if (p.err != 0) {
      if (atomicCAS(&s_err, 0, p.err) == 0) s_info = u;
    }
    my_a += p.new_hp + p.new_lp + (MID ? p.new_mp : 0);
    my_f += p.free_hp + p.free_lp + (MID ? p.free_mp : 0);
  }
  int tot_a, tot_f;
  const int aoff = block_exclusive_scan(my_a, s_warp, &tot_a);
  const int foff = block_exclusive_scan(my_f, s_warp, &tot_f);
  if (threadIdx.x == 0 && s_err == 0 && (unsigned long long)tot_a > end - start) s_err = DKV_ERR_NO_PAGES;
  __syncthreads();
  if (s_err != 0) {
    if (threadIdx.x == 0) latch_error(pv, s_err, s_info);
    return;
  }
  // New pages are read from [start, start+A), inside the free region; freed
  // pages are written to [end, end+F), inside the used region (F <= pages in
  // use), so the two never overlap and one pass suffices.
  int a = aoff, f = foff;
  for (int u = u0; u < u1; u++) {
    const DecodePlan& p = sc.dplan[u];
    const int i = u / pv.hkv, kvh = u % pv.hkv, slot = sa.slots[i];
    int* cn = pv.cnt(layer, slot, kvh);
    int* row = pv.row(layer, slot, kvh);
    // the page counts before the step, from the plan (new = old + new - freed)
    const int php0 = p.php - p.new_hp + p.free_hp, plp0 = p.plp - p.new_lp + p.free_lp;
    const int pmp0 = MID ? p.pmp - p.new_mp + p.free_mp : 0;
    if (p.new_hp) row[php0] = s_list[a++];
    if (p.new_lp) row[pv.L - 1 - plp0] = s_list[a++];
    if (MID && p.new_mp) row[pv.L + pmp0] = s_list[a++];
    if (p.free_hp) {
      pv.list[(end + (unsigned long long)(f++)) % pv.n_pages] = row[php0 - 1];
      row[php0 - 1] = -1;
    }
    if (p.free_lp) {
      pv.list[(end + (unsigned long long)(f++)) % pv.n_pages] = row[pv.L - plp0];
      row[pv.L - plp0] = -1;
    }
    if (MID && p.free_mp) {
      pv.list[(end + (unsigned long long)(f++)) % pv.n_pages] = row[pv.L + pmp0 - 1];
      row[pv.L + pmp0 - 1] = -1;
    }
    cn[0] = p.nh; cn[1] = p.nl; cn[2] = p.php; cn[3] = p.plp;
    if (MID) { cn[4] = p.nm; cn[5] = p.pmp; }
    if (kvh == 0) pv.rq(layer, slot)[2] += 1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    pv.ctl->start = start + (unsigned long long)tot_a;
    pv.ctl->end = end + (unsigned long long)tot_f;
  }
}

// ---------------------------------------------------------------------------
// Request completion: every page of the request (all layers, all KV heads;
// within a head hi pages left to right, then lo pages from the outermost in,
// then mid pages left to right) appended at the list end by one prefix sum;
// rows and state cleared.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kCoordThreads) k_free_request(PoolView pv, int slot) {
  if (pv.noop()) return;
  extern __shared__ int s_dyn[];
  __shared__ int s_warp[32];
  const int n_units = pv.n_layers * pv.hkv;
  int* s_c = s_dyn;             // pages per (layer, KV head) -> exclusive offsets
  int* s_h = s_dyn + n_units;   // hi pages per (layer, KV head)
  int* s_l = s_dyn + 2 * n_units;   // lo pages (three-tier pools: mid pages follow them)
  for (int u = threadIdx.x; u < n_units; u += blockDim.x) {
    const int layer = u / pv.hkv, kvh = u % pv.hkv;
    const int* cn = pv.cnt(layer, slot, kvh);
    const bool act = pv.rq(layer, slot)[0] != 0;
    s_c[u] = act ? cn[2] + cn[3] + (pv.mid_enabled ? cn[5] : 0) : 0;
    s_h[u] = act ? cn[2] : 0;
    s_l[u] = act ? cn[3] : 0;
  }
  __syncthreads();
  const int tot = block_scan_array(s_c, n_units, s_warp);
  const unsigned long long end = pv.ctl->end;
  // page x of the request (in (layer, KV head) order, hi pages then lo pages
  // from the outermost inward) goes to list position end + x; its head is the
  // last u with s_c[u] <= x
  for (int x = threadIdx.x; x < tot; x += blockDim.x) {
    int lo = 0, hi = n_units - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_c[mid] <= x) lo = mid; else hi = mid - 1;
    }
    const int* row = pv.row(lo / pv.hkv, slot, lo % pv.hkv);
    const int k = x - s_c[lo], nh = s_h[lo], nl = s_l[lo];
    pv.list[(end + (unsigned long long)x) % pv.n_pages] =
        k < nh ? row[k] : (k < nh + nl ? row[pv.L - 1 - (k - nh)] : row[pv.L + (k - nh - nl)]);
  }
  __syncthreads();
  for (int u = 0; u < n_units; u++) {
    int* row = pv.row(u / pv.hkv, slot, u % pv.hkv);
    for (int e = threadIdx.x; e < pv.Lrow; e += blockDim.x) row[e] = -1;
  }
  for (int u = threadIdx.x; u < n_units; u += blockDim.x) {
    int* cn = pv.cnt(u / pv.hkv, slot, u % pv.hkv);
    for (int x = 0; x < pv.cstride; x++) cn[x] = 0;
  }
  for (int layer = threadIdx.x; layer < pv.n_layers; layer += blockDim.x) {
    int* rq = pv.rq(layer, slot);
    rq[0] = rq[1] = rq[2] = rq[3] = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) pv.ctl->end = end + (unsigned long long)tot;
}

// ---------------------------------------------------------------------------
cudaError_t launch_setup(const Pool& P, const CallArgs& args, cudaStream_t st) {
  k_setup<<<1, 256, 0, st>>>(P.pv, args);
  return cudaGetLastError();
}

cudaError_t launch_prompt_plan(Pool& P, int layer, int n_req, cudaStream_t st) {
  const int n_units = n_req * P.pv.hkv;
  const int smem = n_units * (int)sizeof(int);
  const int grid = (n_units + kPlanWarps - 1) / kPlanWarps;
  cudaError_t e = launch_dependent(k_prompt_plan_heads, grid, dim3(32 * kPlanWarps), 0, st, P.pv, P.sc);
  if (e != cudaSuccess) return e;
  e = launch_dependent(k_prompt_plan_grant, grid, dim3(32 * kPlanWarps), (size_t)smem, st, P.pv, P.sc);
  if (e != cudaSuccess) return e;
  return launch_dependent(k_prompt_plan_commit, grid, dim3(32 * kPlanWarps), (size_t)smem, st, P.pv, layer, P.sc);
}

cudaError_t configure_alloc() {
  // coordination kernels keep two ints per head in shared memory
  cudaError_t e = cudaFuncSetAttribute(k_prompt_plan_grant, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_prompt_plan_commit, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_free_request, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_decode_alloc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_decode_alloc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
}

// A programmatic dependent of k_decode_plan. One CTA, a thread per head up to
// 1024 (its block-wide scans wait at barriers for every warp of the block).
cudaError_t launch_decode_alloc(Pool& P, int layer, const SlotArgs& sa, cudaStream_t st) {
  const int n_units = sa.n * P.pv.hkv;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(1);
  lc.blockDim = dim3(std::min(kCoordThreads, (n_units + 31) / 32 * 32));
  lc.dynamicSmemBytes = (P.pv.mid_enabled ? 3 : 2) * (size_t)n_units * sizeof(int);   // the list window
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  const cudaError_t e = P.pv.mid_enabled ? cudaLaunchKernelEx(&lc, k_decode_alloc<true>, P.pv, layer, P.sc, sa)
                                         : cudaLaunchKernelEx(&lc, k_decode_alloc<false>, P.pv, layer, P.sc, sa);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_free(Pool& P, int slot, cudaStream_t st) {
  const int smem = 3 * P.pv.n_layers * P.pv.hkv * (int)sizeof(int);
  k_free_request<<<1, kCoordThreads, smem, st>>>(P.pv, slot);
  return cudaGetLastError();
}

}  // namespace dkv
