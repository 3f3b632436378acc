// prompt_tc.cu — the two observation-window passes of prompt-phase scoring
// (DiffKV, compaction policy, prompt phase) on the fifth-generation tensor
// cores: tcgen05 MMAs with fp16 operands staged by TMA tensor copies and fp32
// accumulators in tensor memory.
//
//   a1  lse_{h,p} = log sum_{j<=p} exp(q_{h,p}.k_j / sqrt(d)): D = Q K^T, one
//       accumulator row per (observation query, head), one epilogue thread per
//       row folding the tile's 128 keys into (max, sum) in the log2 domain.
//   a2  S_j = sum_{p>=j} max_h exp(l_{h,p,j} - lse_{h,p}): D = K Q^T, one
//       accumulator row per key, one epilogue thread per key taking the max
//       over the group's heads and the sum over the observation queries.
//
// One persistent CTA per SM takes a contiguous range of the call's (head, key
// tile) pairs, tiles of one head consecutive. Warp 0 issues the TMA copies
// (the head's queries once per head, double-buffered; the key tiles through a
// ring of stages), warp 1 owns the tensor memory and issues the MMAs (two
// accumulators, so that the epilogue of one tile overlaps the MMAs of the
// next), warps 2..5 run the epilogue. Every wait is bounded; on expiry the
// kernel latches DKV_ERR_TIMEOUT, waits (bounded) for its own copies and
// MMAs, frees its tensor memory and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "dkv_kernels.cuh"
#include "dkv_tc.cuh"

namespace dkv {

constexpr int kTcThreads = 320;      // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue
constexpr int kTcEpi = 256;          // epilogue threads: two per accumulator row
constexpr int kTcBarEpi = 1;         // named barrier of the epilogue warps

template <int G>
struct TcCfg {
  static constexpr int MT = (kObs * G + 127) / 128;   // 128-row tiles of the query rows (a1)
  static constexpr int QROWS = 128 * MT;              // query rows a buffer holds
  static constexpr int QBUF = 2 * QROWS * 128;        // one query buffer: two feature halves
  static constexpr int QTX = 2 * kObs * G * 128;      // bytes the two query boxes deliver
  static constexpr int KS = G <= 4 ? 4 : 2;           // key-tile stages
  static constexpr int KBUF = 2 * kKeyBlock * 128;    // one key tile: two feature halves
  static constexpr int ACC = 128 * MT;                // tensor-memory columns per accumulator
  static constexpr int TCOLS = 2 * ACC;               // two accumulators
  // shared memory after the 1024-byte alignment pad
  static constexpr int OFF_K = 2 * QBUF;
  static constexpr int OFF_MISC = OFF_K + KS * KBUF;
};

template <int G>
static int tc_smem_bytes(int n_req) {
  return 1024 + TcCfg<G>::OFF_MISC + 8 * (2 * TcCfg<G>::KS + 8) + 16 + 4 * (n_req + 1) + 4 * kObs * G + 64 +
         8 * 2 * 2 * 128 + 16;
}

// lse2[unit][h*32 + o] = m + log2(l) over the key tiles' partials (log2
// domain); -inf for observation rows with a negative position. A warp per
// row: lane k folds the partials of tiles k, k + 32, ... (their loads all in
// flight at once), then the lanes combine by shuffles. Grid: (unit, row group
// of kMergeWarps rows).
constexpr int kMergeWarps = 8;
__global__ void __launch_bounds__(32 * kMergeWarps) k_prompt_lse_merge(PoolView pv, const float2* __restrict__ partial,
                                                                       float* lse2, int nkb_cap) {
  if (!dependent_begin(pv)) return;
  const int unit = blockIdx.x, i = unit / pv.hkv;
  const int rows = kObs * pv.G;
  const int r = blockIdx.y * kMergeWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= rows) return;
  const int n0 = pv.call->lens[i];
  const int nkb = (n0 + kKeyBlock - 1) / kKeyBlock;
  const float2* src = partial + (size_t)unit * nkb_cap * rows + r;
  float m = -INFINITY, l = 0.0f;
  for (int kb = lane; kb < nkb; kb += 32) {
    const float2 pl = __ldcg(src + (size_t)kb * rows);
    const float mn = fmaxf(m, pl.x);
    if (mn == -INFINITY) continue;
    l = l * exp2f(m - mn) + pl.y * exp2f(pl.x - mn);
    m = mn;
  }
  float M = m;
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, s));
  float L = M == -INFINITY || m == -INFINITY ? 0.0f : l * exp2f(m - M);
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) L += __shfl_xor_sync(0xffffffffu, L, s);
  if (lane == 0) lse2[(size_t)unit * rows + r] = (L > 0.0f) ? M + log2f(L) : -INFINITY;
}

// SCORE = false: a1 (partial max and sum per query row and key tile).
// SCORE = true: a2 (the scores; tiers and ranks follow from them in
// k_prompt_given, the classification of the CUDA-core path).
template <int G, bool SCORE>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_prompt_tc(PoolView pv, const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tq,
                const float* __restrict__ lse2, float2* partial, float* score_out, int nkb_cap) {
  using C = TcCfg<G>;
  if (!dependent_begin(pv)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_MISC);
  // barriers: kfull[KS], kempty[KS], qfull[2], qempty[2], afull[2], aempty[2]
  const uint32_t b0 = smem_u32(bars);
  auto kfull = [&](int s) { return b0 + 8u * s; };
  auto kempty = [&](int s) { return b0 + 8u * (C::KS + s); };
  auto qfull = [&](int b) { return b0 + 8u * (2 * C::KS + b); };
  auto qempty = [&](int b) { return b0 + 8u * (2 * C::KS + 2 + b); };
  auto afull = [&](int b) { return b0 + 8u * (2 * C::KS + 4 + b); };
  auto aempty = [&](int b) { return b0 + 8u * (2 * C::KS + 6 + b); };
  uint32_t* s_taddr = reinterpret_cast<uint32_t*>(bars + 2 * C::KS + 8);
  int* s_fail = reinterpret_cast<int*>(s_taddr + 1);
  int* s_cnt = s_fail + 1;                              // [16] scan scratch
  int* s_roff = s_cnt + 16;                             // [n_req + 1] first tile of each request
  const CallArgs* ca = pv.call;
  const int n_req = ca->n_req, hkv = pv.hkv;
  float* s_lse = reinterpret_cast<float*>(s_roff + n_req + 1);   // [32 G] lse2 of the current head (a2)
  // [2][MT][128] partial (max, sum) of the second epilogue half (a1), or
  // [2][128] partial scores (a2), by accumulator
  float2* s_half = reinterpret_cast<float2*>(
      (reinterpret_cast<uintptr_t>(s_lse + kObs * G) + 15) & ~uintptr_t(15));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // tiles of the call: request i holds hkv heads x nkb(i) key tiles
  {
    const int per = (n_req + kTcThreads - 1) / kTcThreads;
    const int r0 = min(n_req, (int)threadIdx.x * per), r1 = min(n_req, r0 + per);
    int sum = 0;
    for (int r = r0; r < r1; r++) sum += (ca->lens[r] + kKeyBlock - 1) / kKeyBlock * hkv;
    // exclusive scan of the per-thread sums over the block (6 warps)
    int x = sum;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, s);
      if (lane >= s) x += y;
    }
    if (lane == 31) s_cnt[warp] = x;
    __syncthreads();
    int run = x - sum;
    for (int w = 0; w < warp; w++) run += s_cnt[w];
    for (int r = r0; r < r1; r++) {
      s_roff[r] = run;
      run += (ca->lens[r] + kKeyBlock - 1) / kKeyBlock * hkv;
    }
    if (threadIdx.x == kTcThreads - 1) s_roff[n_req] = run;
    __syncthreads();
  }
  const int total = s_roff[n_req];
  const int t0 = (int)((long long)total * blockIdx.x / gridDim.x);
  const int t1 = (int)((long long)total * (blockIdx.x + 1) / gridDim.x);
  if (t0 >= t1) return;
  // (request, head, key tile) of tile t, walking forward from the previous one
  struct Tile {
    int i, kvh, kb, nkb;
  };
  auto locate = [&](int t) {
    int lo = 0, hi = n_req - 1;   // last request with s_roff <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_roff[mid] <= t) lo = mid; else hi = mid - 1;
    }
    Tile x;
    x.i = lo;
    x.nkb = (ca->lens[lo] + kKeyBlock - 1) / kKeyBlock;
    const int off = t - s_roff[lo];
    x.kvh = off / x.nkb;
    x.kb = off % x.nkb;
    return x;
  };
  // a1 walks the range forward, a2 backward: the key tiles a1 read last are
  // the ones still in L2 when a2 starts
  auto next = [&](Tile& x) {
    if (!SCORE) {
      if (++x.kb == x.nkb) {
        x.kb = 0;
        if (++x.kvh == hkv) {
          x.kvh = 0;
          x.i++;
          x.nkb = x.i < n_req ? (ca->lens[x.i] + kKeyBlock - 1) / kKeyBlock : 1;
        }
      }
    } else if (--x.kb < 0) {
      if (--x.kvh < 0) {
        x.kvh = hkv - 1;
        x.i--;
        x.nkb = x.i >= 0 ? (ca->lens[x.i] + kKeyBlock - 1) / kKeyBlock : 1;
      }
      x.kb = x.nkb - 1;
    }
  };
  const int t_first = SCORE ? t1 - 1 : t0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::KS; s++) {
      mbar_init(kfull(s), 1);
      mbar_init(kempty(s), 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(qfull(b), 1);
      mbar_init(qempty(b), 1);
      mbar_init(afull(b), 1);
      mbar_init(aempty(b), kTcEpi);
    }
    *s_fail = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(s_taddr), C::TCOLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *s_taddr;
  auto fail = [&](int where) {
    if (atomicCAS(&pv.ctl->error, 0, DKV_ERR_TIMEOUT) == 0) pv.ctl->error_info = where;
    *(volatile int*)s_fail = 1;
  };
  auto failed = [&]() { return *(volatile int*)s_fail != 0; };

  if (warp == 0) {
    // ---- producer: the head's queries on a head change, then the key tile ----
    if (lane == 0) {
      Tile x = locate(t_first);
      int qi = 0, prev_unit = -1, last_s[8], last_q[2];
      for (int s = 0; s < 8; s++) last_s[s] = -1;
      last_q[0] = last_q[1] = -1;
      for (int it = 0; it < t1 - t0 && !failed(); it++, next(x)) {
        const int unit = x.i * hkv + x.kvh;
        if (unit != prev_unit) {
          const int b = qi & 1;
          if (qi >= 2 && !mbar_wait_bounded(qempty(b), ((qi >> 1) - 1) & 1)) { fail(1); break; }
          mbar_expect_tx(qfull(b), C::QTX);
          uint8_t* qb = smem + b * C::QBUF;
          for (int h = 0; h < 2; h++)
            tma_load_4d(smem_u32(qb + h * C::QROWS * 128), &tq, 64 * h, x.kvh * G, 0, x.i, qfull(b));
          last_q[b] = qi;
          qi++;
          prev_unit = unit;
        }
        const int s = it % C::KS;
        if (it >= C::KS && !mbar_wait_bounded(kempty(s), ((it / C::KS) - 1) & 1)) { fail(2); break; }
        mbar_expect_tx(kfull(s), C::KBUF);
        uint8_t* kbuf = smem + C::OFF_K + s * C::KBUF;
        const int row0 = (int)(ca->tok0[x.i] + (long long)x.kb * kKeyBlock);
        for (int h = 0; h < 2; h++)
          tma_load_3d(smem_u32(kbuf + h * kKeyBlock * 128), &tk, 64 * h, x.kvh, row0, kfull(s));
        last_s[s] = it;
      }
      // no copy of this CTA may still be in flight when it exits
      for (int s = 0; s < C::KS; s++)
        if (last_s[s] >= 0) mbar_wait_bounded(kfull(s), (last_s[s] / C::KS) & 1);
      for (int b = 0; b < 2; b++)
        if (last_q[b] >= 0) mbar_wait_bounded(qfull(b), (last_q[b] >> 1) & 1);
    }
  } else if (warp == 1) {
    // ---- MMA issuer ----
    if (lane == 0) {
      Tile x = locate(t_first);
      int qi = -1, prev_unit = -1, issued = -1;
      for (int it = 0; it < t1 - t0 && !failed(); it++) {
        const int unit = x.i * hkv + x.kvh;
        if (unit != prev_unit) {
          qi++;
          if (!mbar_wait_bounded(qfull(qi & 1), (qi >> 1) & 1)) { fail(3); break; }
          prev_unit = unit;
        }
        const int s = it % C::KS, ab = it & 1;
        if (!mbar_wait_bounded(kfull(s), (it / C::KS) & 1)) { fail(4); break; }
        if (it >= 2 && !mbar_wait_bounded(aempty(ab), ((it >> 1) - 1) & 1)) { fail(5); break; }
        tc_fence_after();
        const uint32_t qs = smem_u32(smem + (qi & 1) * C::QBUF);
        const uint32_t ks = smem_u32(smem + C::OFF_K + s * C::KBUF);
        const uint32_t d = tbase + ab * C::ACC;
#pragma unroll
        for (int k = 0; k < 8; k++) {
          const uint32_t kq = (k >> 2) * C::QROWS * 128 + (k & 3) * 32;    // feature half, 16-feature step
          const uint32_t kk = (k >> 2) * kKeyBlock * 128 + (k & 3) * 32;
          if (SCORE) {
            umma_f16(d, umma_desc_sw128(ks + kk), umma_desc_sw128(qs + kq), umma_idesc_f16(128, kObs * G), k > 0);
          } else {
#pragma unroll
            for (int mt = 0; mt < C::MT; mt++)
              umma_f16(d + 128 * mt, umma_desc_sw128(qs + kq + mt * 128 * 128), umma_desc_sw128(ks + kk),
                       umma_idesc_f16(128, kKeyBlock), k > 0);
          }
        }
        umma_commit(kempty(s));
        next(x);
        const bool last_of_head = it + 1 == t1 - t0 || x.i * hkv + x.kvh != unit;
        if (last_of_head) umma_commit(qempty(qi & 1));
        umma_commit(afull(ab));
        issued = it;
      }
      // every MMA of this CTA has completed before it exits
      if (issued >= 0) mbar_wait_bounded(afull(issued & 1), (issued >> 1) & 1);
    }
  } else {
    // ---- epilogue: warps 2..9; thread = accumulator row (lane group warp % 4)
    // and half hf of the row's columns ----
    const int lg = warp & 3, row = 32 * lg + lane, hf = (warp - 2) >> 2;
    const uint32_t tl = tbase + ((uint32_t)(32 * lg) << 16);
    const float sc = 1.4426950408889634f * rsqrtf((float)kD);
    Tile x = locate(t_first);
    int lse_unit = -1;
    // a2 with G <= 4: -lse2 of this thread's 16 G columns held in registers
    constexpr bool kLseReg = G <= 4;
    float nlse[kLseReg ? kObs / 2 * G : 1];
    for (int it = 0; it < t1 - t0; it++, next(x)) {
      const int ab = it & 1;
      // on expiry the tile still runs through its barriers (with whatever the
      // accumulator holds); the combine barrier below makes one decision for
      // all epilogue threads, so that none is left waiting at a barrier
      const bool ok = mbar_wait_bounded(afull(ab), (it >> 1) & 1);
      if (!ok) fail(6);
      tc_fence_after();
      const int i = x.i, n0 = ca->lens[i], key0 = x.kb * kKeyBlock;
      const int unit = i * hkv + x.kvh;
      if (!SCORE) {
        // keys 64 hf .. 64 hf + 63 of the row: max first, then one exp2 each;
        // eight independent partial maxima and sums keep the chains short
        constexpr int NK = kKeyBlock / 2;
        float m[C::MT], l[C::MT];
        const bool full = key0 + kKeyBlock - 1 <= n0 - kObs;    // no key after any query row's position
#pragma unroll
        for (int mt = 0; mt < C::MT; mt++) {
          const int r = 128 * mt + row;                  // query row (o, h): r = o G + h
          const int p = n0 - kObs + r / G;               // its position
          const int kc = key0 + NK * hf;                 // first key of the half
          float v[NK];
#pragma unroll
          for (int c0 = 0; c0 < NK; c0 += 32) tmem_ld32_nowait(tl + ab * C::ACC + 128 * mt + NK * hf + c0, v + c0);
          tmem_wait_ld();
          if (mt == C::MT - 1) {
            tc_fence_before();
            mbar_arrive(aempty(ab));                     // the accumulator is free for the MMA after next
          }
          if (!full) {
#pragma unroll
            for (int e = 0; e < NK; e++)
              if (kc + e > p) v[e] = -INFINITY;
          }
          float pm[8];
#pragma unroll
          for (int e = 0; e < 8; e++) pm[e] = v[e];
#pragma unroll
          for (int e = 8; e < NK; e++) pm[e & 7] = fmaxf(pm[e & 7], v[e]);
          const float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                                 fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
          m[mt] = mx * sc;                               // sc > 0: the max commutes with the scale
          l[mt] = 0.0f;
          if (mx != -INFINITY) {
            float ps[8];
#pragma unroll
            for (int e = 0; e < 8; e++) ps[e] = 0.0f;
#pragma unroll
            for (int e = 0; e < NK; e++) ps[e & 7] += fast_exp2(__fmaf_rn(v[e], sc, -m[mt]));
            l[mt] = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
          }
        }
        // the two halves of each row combine in the first half
        float2* hb = s_half + ab * C::MT * 128;
        if (hf == 1) {
#pragma unroll
          for (int mt = 0; mt < C::MT; mt++) hb[mt * 128 + row] = make_float2(m[mt], l[mt]);
        }
        if (!named_all(kTcBarEpi, kTcEpi, ok && !failed())) break;
        if (hf == 0) {
#pragma unroll
          for (int mt = 0; mt < C::MT; mt++) {
            const int r = 128 * mt + row;
            if (r < kObs * G) {
              const float2 o2 = hb[mt * 128 + row];
              const float mn = fmaxf(m[mt], o2.x);
              float lt = 0.0f;
              if (mn != -INFINITY) lt = l[mt] * fast_exp2(m[mt] - mn) + o2.y * fast_exp2(o2.x - mn);
              const int o = r / G, h = r % G;
              partial[((size_t)unit * nkb_cap + x.kb) * (kObs * G) + h * kObs + o] = make_float2(mn, lt);
            }
          }
        }
      } else {
        if (unit != lse_unit) {                          // lse2 of the head's query rows
          named_sync(kTcBarEpi, kTcEpi);                 // the previous head's values are no longer read
          for (int r = threadIdx.x - 64; r < kObs * G; r += kTcEpi) s_lse[r] = lse2[(size_t)unit * kObs * G + r];
          named_sync(kTcBarEpi, kTcEpi);
          if (kLseReg) {
#pragma unroll
            for (int c = 0; c < (kLseReg ? kObs / 2 * G : 1); c++)
              nlse[c] = -s_lse[(c % G) * kObs + kObs / 2 * hf + c / G];
          }
          lse_unit = unit;
        }
        const int j = key0 + row;
        const bool full = j <= n0 - kObs;                // the key precedes every observation query
        // observation queries 16 hf .. 16 hf + 15: columns (o, h) = o G + h,
        // the max over the heads of one query, then one exp2 per query into
        // four partial sums
        constexpr int NC = kObs / 2 * G;                 // columns of a half
        const int cbase = NC * hf;
        float ps[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        float y = -INFINITY;
#pragma unroll
        for (int c0 = 0; c0 < NC; c0 += 64) {
          constexpr int W = NC < 64 ? NC : 64;
          float v[W];
#pragma unroll
          for (int c = 0; c < W; c += 16)
            if (c0 + c < NC) tmem_ld16_nowait(tl + ab * C::ACC + cbase + c0 + c, v + c);
          tmem_wait_ld();
          if (c0 + W >= NC) {
            tc_fence_before();
            mbar_arrive(aempty(ab));
          }
#pragma unroll
          for (int e = 0; e < W; e++) {
            const int col = c0 + e, o = col / G, h = col % G;    // o relative to the half
            if (col >= NC) break;
            const int og = kObs / 2 * hf + o;
            y = fmaxf(y, __fmaf_rn(v[e], sc, kLseReg ? nlse[col] : -s_lse[h * kObs + og]));
            if (h == G - 1) {
              if (full || j <= n0 - kObs + og) ps[o & 3] += fast_exp2(y);
              y = -INFINITY;
            }
          }
        }
        const float sh = (ps[0] + ps[1]) + (ps[2] + ps[3]);
        float* hb = reinterpret_cast<float*>(s_half) + ab * 128;
        if (hf == 1) hb[row] = sh;
        if (!named_all(kTcBarEpi, kTcEpi, ok && !failed())) break;
        if (hf == 0 && j < n0) score_out[(size_t)(ca->tok0[i] + j) * hkv + x.kvh] = sh + hb[row];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, C::TCOLS);
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps of the call's keys and observation queries, launch.
// ---------------------------------------------------------------------------
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_encode_mu;

cudaError_t encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::lock_guard<std::mutex> lock(g_encode_mu);
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !p) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  *fn = g_encode;
  return cudaSuccess;
}

// keys [n_tok][hkv][128] fp16: box = 128 tokens x one head x 64 features
// queries [n_req][32][hkv G][128] fp16: box = 32 queries x G heads x 64 features
cudaError_t make_maps(const Pool& P, const __half* k, const __half* q_obs, long long n_tok, int n_req,
                      CUtensorMap* mk, CUtensorMap* mq) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  cudaError_t e = encoder(&enc);
  if (e != cudaSuccess) return e;
  const int hkv = P.pv.hkv, G = P.pv.G, hq = hkv * G;
  const cuuint32_t es[4] = {1, 1, 1, 1};
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)hkv, (cuuint64_t)n_tok};
    const cuuint64_t str[2] = {(cuuint64_t)kD * 2, (cuuint64_t)hkv * kD * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)kKeyBlock};
    if (enc(mk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half*>(k), dims, str, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)hq, (cuuint64_t)kObs, (cuuint64_t)n_req};
    const cuuint64_t str[3] = {(cuuint64_t)kD * 2, (cuuint64_t)hq * kD * 2, (cuuint64_t)kObs * hq * kD * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)kObs, 1};
    if (enc(mq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<__half*>(q_obs), dims, str, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

template <int G>
cudaError_t launch_tc_g(Pool& P, const CUtensorMap& mk, const CUtensorMap& mq, const float* lse_obs, int n_req,
                        float* score_out, cudaStream_t st) {
  const Scratch& s = P.sc;
  const int smem = tc_smem_bytes<G>(n_req);
  if (lse_obs)                    // the prompt's attention left the log-sum-exps: a2 alone
    return launch_dependent(k_prompt_tc<G, true>, dim3(P.sm_count), dim3(kTcThreads), (size_t)smem, st, P.pv, mk,
                            mq, lse_obs, (float2*)nullptr, score_out, s.nkb_cap);
  cudaError_t e = launch_dependent(k_prompt_tc<G, false>, dim3(P.sm_count), dim3(kTcThreads), (size_t)smem, st, P.pv,
                                   mk, mq, (const float*)nullptr, s.partial, (float*)nullptr, s.nkb_cap);
  if (e != cudaSuccess) return e;
  e = launch_dependent(k_prompt_lse_merge, dim3(n_req * P.pv.hkv, (kObs * P.pv.G + kMergeWarps - 1) / kMergeWarps),
                       dim3(32 * kMergeWarps), 0, st, P.pv, (const float2*)s.partial, s.lse2, s.nkb_cap);
  if (e != cudaSuccess) return e;
  return launch_dependent(k_prompt_tc<G, true>, dim3(P.sm_count), dim3(kTcThreads), (size_t)smem, st, P.pv, mk, mq,
                          (const float*)s.lse2, (float2*)nullptr, score_out, s.nkb_cap);
}

template <int G>
cudaError_t configure_tc_g() {
  const int smem = tc_smem_bytes<G>(kMaxCallReq);
  cudaError_t e = cudaFuncSetAttribute(k_prompt_tc<G, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_prompt_tc<G, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}
}  // namespace

// The driver's tensor-map encoder, looked up once (shared with prefill_tc.cu).
cudaError_t tma_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) { return encoder(fn); }

cudaError_t configure_prompt_tc() {
  cudaError_t e;
  if ((e = configure_tc_g<1>()) != cudaSuccess) return e;
  if ((e = configure_tc_g<2>()) != cudaSuccess) return e;
  if ((e = configure_tc_g<3>()) != cudaSuccess) return e;
  if ((e = configure_tc_g<4>()) != cudaSuccess) return e;
  if ((e = configure_tc_g<5>()) != cudaSuccess) return e;
  if ((e = configure_tc_g<6>()) != cudaSuccess) return e;
  if ((e = configure_tc_g<7>()) != cudaSuccess) return e;
  return configure_tc_g<8>();
}

// a1, the partial merge and a2 of one prompt call on the tensor cores (a2
// alone when the log-sum-exps are given).
cudaError_t launch_scoring_tc(Pool& P, const __half* k, const __half* q_obs, const float* lse_obs, long long n_tok,
                              int n_req, float* score_out, cudaStream_t st) {
  CUtensorMap mk, mq;
  cudaError_t e = make_maps(P, k, q_obs, n_tok, n_req, &mk, &mq);
  if (e != cudaSuccess) return e;
  switch (P.pv.G) {
    case 1: return launch_tc_g<1>(P, mk, mq, lse_obs, n_req, score_out, st);
    case 2: return launch_tc_g<2>(P, mk, mq, lse_obs, n_req, score_out, st);
    case 3: return launch_tc_g<3>(P, mk, mq, lse_obs, n_req, score_out, st);
    case 4: return launch_tc_g<4>(P, mk, mq, lse_obs, n_req, score_out, st);
    case 5: return launch_tc_g<5>(P, mk, mq, lse_obs, n_req, score_out, st);
    case 6: return launch_tc_g<6>(P, mk, mq, lse_obs, n_req, score_out, st);
    case 7: return launch_tc_g<7>(P, mk, mq, lse_obs, n_req, score_out, st);
    default: return launch_tc_g<8>(P, mk, mq, lse_obs, n_req, score_out, st);
  }
}

}  // namespace dkv
