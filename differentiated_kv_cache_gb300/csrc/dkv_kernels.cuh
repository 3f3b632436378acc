// dkv_kernels.cuh — internal interface between the C-ABI host code (pool.cu)
// and the kernel files (prompt.cu, alloc.cu, decode_compact.cu, attention.cu).
#pragma once

#include <vector>

#include "dkv_common.cuh"

namespace dkv {

constexpr int kKeyBlock = 128;     // prompt tokens per scoring / classification block
constexpr int kChunk = 16;         // decode-attention tokens per mma chunk
constexpr int kAttnWarps = 4;      // warps per decode-attention CTA
constexpr int kVictimWarps = 8;    // warps of an attention epilogue block, each leaving a victim-key partial
// Decode-attention scratch row per 16-slot chunk (floats): the log2-domain
// logits [query < G][16 slots]; the epilogue takes the scores before the
// update and the page IDs from the pages themselves.

// One slot write of a generation-phase step.
// src: the new token, or a stored token of tier src_tier at slot src_slot,
// re-quantised when src_tier differs from dst_tier (a demotion) and copied
// as is otherwise.
enum MoveSrc { kSrcNew = 0, kSrcDemote = 1 };
struct Move {
  int dst_tier, dst_slot, src, src_slot;
  int src_tier;
};
// Per-head plan of one generation-phase step (written by k_decode_plan).
struct DecodePlan {
  int nh, nl;                          // token counts after the step
  int php, plp;                        // page counts after the step
  int new_hp, new_lp, free_hp, free_lp;
  int n_moves, err;
  Move mv[3];
  int nm, pmp, new_mp, free_mp;        // the mid tier (three-tier pools), as above
};

// Argmin over tokens of (importance, position): key = order_key(importance)
// << 32 | position, unique within a head; smaller wins (ties in importance go
// to the smaller position).
struct ArgMin {
  unsigned long long key;
  int slot;
};
__device__ __forceinline__ ArgMin amin(ArgMin a, ArgMin b) { return b.key < a.key ? b : a; }
__device__ __forceinline__ ArgMin shfl_amin(ArgMin a, int s) {
  ArgMin b;
  b.key = __shfl_xor_sync(0xffffffffu, a.key, s);
  b.slot = __shfl_xor_sync(0xffffffffu, a.slot, s);
  return amin(a, b);
}

// Block-wide argmin of two keys at once (s_tmp: two entries per warp); every
// thread returns with both results.
__device__ __forceinline__ void block_amin2(ArgMin& a, ArgMin& b, ArgMin* s_tmp) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    a = shfl_amin(a, s);
    b = shfl_amin(b, s);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (lane == 0) {
    s_tmp[warp] = a;
    s_tmp[nw + warp] = b;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < nw; w++) {
      a = amin(a, s_tmp[w]);
      b = amin(b, s_tmp[nw + w]);
    }
    s_tmp[0] = a;
    s_tmp[nw] = b;
  }
  __syncthreads();
  a = s_tmp[0];
  b = s_tmp[nw];
}

// Block-wide argmin of three keys at once (s_tmp: three entries per warp).
__device__ __forceinline__ void block_amin3(ArgMin& a, ArgMin& b, ArgMin& c, ArgMin* s_tmp) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    a = shfl_amin(a, s);
    b = shfl_amin(b, s);
    c = shfl_amin(c, s);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (lane == 0) {
    s_tmp[warp] = a;
    s_tmp[nw + warp] = b;
    s_tmp[2 * nw + warp] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < nw; w++) {
      a = amin(a, s_tmp[w]);
      b = amin(b, s_tmp[nw + w]);
      c = amin(c, s_tmp[2 * nw + w]);
    }
    s_tmp[0] = a;
    s_tmp[nw] = b;
    s_tmp[2 * nw] = c;
  }
  __syncthreads();
  a = s_tmp[0];
  b = s_tmp[nw];
  c = s_tmp[2 * nw];
}

// One stored token's part in the victim search of the next generation step
// (length n = N + 1 after its append, update count upd): its importance
// S / c and argmin key; hi tokens before wlim = n - W are hi-victim
// candidates, the hi token at pc = n - W - 1 is t_c, every lo token is a
// lo-victim candidate.
// In a three-tier pool every mid token is a mid-victim candidate (bm).
__device__ __forceinline__ void victim_token(float score, int pos, int slot, int tier, int n0, int upd, int pc,
                                             int wlim, ArgMin& bh, ArgMin& bl, ArgMin& bm, int& xc, float& ic) {
  const float imp = __fdiv_rn(score, (float)score_count(pos, n0, upd));
  const unsigned long long key = ((unsigned long long)order_key(imp) << 32) | (uint32_t)pos;
  if (tier == kTierHi) {
    if (pos == pc) {
      xc = slot;
      ic = imp;
    }
    if (pos < wlim) bh = amin(bh, ArgMin{key, slot});
  } else if (tier == kTierLo) {
    bl = amin(bl, ArgMin{key, slot});
  } else {
    bm = amin(bm, ArgMin{key, slot});
  }
}

// Device scratch owned by the pool (sizes fixed at creation).
struct Scratch {
  // prompt
  float2* partial;      // [units][nkb_cap][32*G]
  float* lse2;          // [units][32*G]
  float* score;         // [max_tokens][Hkv]
  uint16_t* tokinfo;    // [max_tokens][Hkv]: rank << 2 | tier
  int2* bcnt;           // [units][nkb_cap]: hi and lo tokens of a key block
  int2* bbase;          // [units][nkb_cap]: their exclusive prefixes over the head's blocks
  int* bcnt_m;          // [units][nkb_cap]: mid tokens of a key block (three-tier pools)
  int* bbase_m;         // [units][nkb_cap]: their exclusive prefixes
  int* rank2pos;        // [units][2 or 3][max_seq]: maps lo, hi (, mid)
  int4* unit_info;      // [units]: grant pages, hi count, lo count, reclaimed pages
  int* unit_mid;        // [units]: mid count (three-tier pools)
  int* grant_ids;       // [units][grant_cap]
  unsigned long long* pbase;   // prompt coordination: list start, end and grant total at the call
  // decode compaction
  DecodePlan* dplan;    // [units]
  ScanPart* dscan;      // [units][max_scan] partials of the generation-phase scan
  int* darrive;         // [units] scan CTAs arrived (zero between calls)
  // decode attention
  float* apart;         // [units][max_splits][G*(128+2)]
  float* alogit;        // [units][max_chunks][G * 16]: per chunk logits
  float* alse;          // [units][G]
  int nkb_cap, grant_cap, max_splits, max_chunks, max_scan;
};

// Host side of a pool.
struct Pool {
  dkv_config cfg;
  int device;
  int sm_count;
  PoolView pv;           // device pointers + geometry
  Scratch sc;
  std::vector<void*> allocations;
  // host mirror of request state: [layer][slot]
  std::vector<int> h_active, h_n0, h_n;
  // device address of the static array of the allocation-free attention
  // entry point on this pool's device (looked up at creation)
  void* static_base = nullptr;
};

// Launchers (return the first CUDA error, cudaSuccess otherwise).
cudaError_t launch_setup(const Pool& P, const CallArgs& args, cudaStream_t st);
// lse_obs: the observation rows' base-2 log-sum-exps from the prompt's own
// attention ([n_req][Hq][32]); null: the score pass computes them itself.
cudaError_t launch_prompt(Pool& P, int layer, int n_req, int max_len, long long n_tok, const __half* k,
                          const __half* v, const __half* q_obs, const float* lse_obs, const float* scores_in,
                          float* scores_out, cudaStream_t st);
// Causal prompt attention of a call (prefill.cu).
cudaError_t launch_prefill(Pool& P, const CallArgs& args, int max_len, const __half* q, const __half* k,
                           const __half* v, float* out, float* lse_obs, cudaStream_t st);
cudaError_t launch_decode(Pool& P, int layer, const SlotArgs& sa, const __half* k, const __half* v,
                          cudaStream_t st);
cudaError_t launch_attention(Pool& P, int layer, const SlotArgs& sa, int max_tokens, const __half* q,
                             float* out, int update_scores, cudaStream_t st);
cudaError_t launch_free(Pool& P, int slot, cudaStream_t st);
// Allocation-free attention: bytes of the static array one call needs, and
// the launcher over that array (attention.cu).
size_t attention_static_bytes(const Pool& P, int n_units, int max_tokens, int update_scores);
cudaError_t static_scratch_address(void** base);
cudaError_t launch_attention_static(Pool& P, int layer, const SlotArgs& sa, int max_tokens, const __half* q,
                                    float* out, int update_scores, cudaStream_t st);
cudaError_t configure_kernels();

// Prologue of a kernel launched as a programmatic dependent (small grids:
// one status read per block): let the next kernel of the chain launch, skip
// on an earlier error, then wait for the kernel before (griddepcontrol.wait)
// ahead of any read of what it wrote, and re-read the status it may have set.
// Called by every thread of the block. LATE: let the next kernel launch only
// after the wait, when it reads before its own wait what kernels before this
// one wrote.
template <bool LATE = false>
__device__ __forceinline__ bool dependent_begin(const PoolView& pv) {
  __shared__ int s_stop;
  if (!LATE) pdl_launch_dependents();
  if (pv.noop()) return false;
  pdl_wait();
  if (LATE) pdl_launch_dependents();
  if (threadIdx.x == 0) s_stop = pv.noop_after_wait() ? 1 : 0;
  __syncthreads();
  return s_stop == 0;
}

// Launch `kernel` as a programmatic dependent of the kernel before it on the
// stream (its blocks may become resident while that kernel drains; the
// kernel itself starts with dependent_begin).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                    Args... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&lc, kernel, args...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dkv
