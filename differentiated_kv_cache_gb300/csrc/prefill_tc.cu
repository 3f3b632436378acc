// prefill_tc.cu — causal GQA attention over the prompt on the fifth-generation
// tensor cores: the model's own attention that DiffKV's compactor follows
// (DiffKV, system implementation: architecture overview; background: the
// attention equation). The last 32 query rows also leave their base-2
// log-sum-exps, which the prompt score pass takes instead of its own pass
// over the keys (dkv_compact_step_prefilled).
//
// One CTA per (128 query rows, query head, prompt), heaviest query tiles
// first. Warp 0 issues the TMA copies (the CTA's queries once; 128-key K and
// V tiles through two stages each), warp 1 issues the MMAs, warps 2..5 run
// the softmax with one thread per query row:
//   S_j = Q K_j^T   tcgen05, A and B from shared memory, D in tensor memory
//                   (three S buffers of 128 columns, so that QK of tile j+1
//                   runs while the softmax of tile j and PV of tile j-1 do)
//   P_j             exp2 of the base-2 logits against a lazily raised row
//                   maximum (O is rescaled only when a row's maximum rises
//                   by more than 2^8), written back over S_j as an fp16 pair
//                   and its fp16 residual (about 22 significant bits)
//   O += P_j V_j    tcgen05 with A = P_j read from tensor memory and B = V_j
//                   MN-major from shared memory, twice (pair and residual)
// The softmax threads read O out of tensor memory at the end. Every wait is
// bounded; on expiry the kernel latches DKV_ERR_TIMEOUT, waits (bounded) for
// its own copies and MMAs, frees its tensor memory and returns.
#include <cudaTypedefs.h>

#include "dkv_kernels.cuh"
#include "dkv_tc.cuh"

namespace dkv {

cudaError_t tma_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn);

constexpr int kPfT = 128;                  // query rows per CTA, keys per tile
constexpr int kPfThreads = 192;            // warp 0 TMA, warp 1 MMA, warps 2..5 softmax
constexpr int kPfHalf = kPfT * 128;        // one 64-feature half of a 128-row fp16 tile: 16 KB
constexpr int kPfTile = 2 * kPfHalf;       // 32 KB
constexpr int kPfStages = 2;
constexpr int kPfOffK = kPfTile;                           // after Q
constexpr int kPfOffV = kPfOffK + kPfStages * kPfTile;
constexpr int kPfOffBar = kPfOffV + kPfStages * kPfTile;
constexpr int kPfSmem = 1024 + kPfOffBar + 256;
constexpr int kPfSBufs = 3;                                // S / P buffers in tensor memory
constexpr uint32_t kPfOCol = kPfSBufs * 128;               // O after them
constexpr uint32_t kPfCols = 512;
constexpr float kPfLazy = 8.0f;                            // probabilities stay below 2^8

struct PrefillTcArgs {
  float* out;       // [tokens][Hq][128]
  float* lse_obs;   // [n_req][Hq][32] or null
};

__global__ void __launch_bounds__(kPfThreads, 1)
    k_prefill_tc(PoolView pv, const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, PrefillTcArgs a, const __grid_constant__ CallArgs ca) {
  if (pv.noop()) return;
  const int hq = blockIdx.y, i = blockIdx.z;
  const int G = pv.G, Hq = pv.hkv * G, kvh = hq / G;
  const int n0 = ca.lens[i];
  const int ntiles = (n0 + kPfT - 1) / kPfT;
  if ((int)blockIdx.x >= ntiles) return;
  const int qt = ntiles - 1 - (int)blockIdx.x;   // heaviest tiles first
  const int r0 = qt * kPfT, nkt = qt + 1;       // key tiles 0 .. qt
  const long long t0 = ca.tok0[i];
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPfOffBar);
  const uint32_t b0 = smem_u32(bars);
  // qfull, kfull[2], kempty[2], vfull[2], vempty[2], sfull[3], pfull[3], pvdone[3], ofull
  const uint32_t qfull = b0, ofull = b0 + 8u * 18;
  auto kfull = [&](int s) { return b0 + 8u * (1 + s); };
  auto kempty = [&](int s) { return b0 + 8u * (3 + s); };
  auto vfull = [&](int s) { return b0 + 8u * (5 + s); };
  auto vempty = [&](int s) { return b0 + 8u * (7 + s); };
  auto sfull = [&](int b) { return b0 + 8u * (9 + b); };
  auto pfull = [&](int b) { return b0 + 8u * (12 + b); };
  auto pvdone = [&](int b) { return b0 + 8u * (15 + b); };
  uint32_t* s_taddr = reinterpret_cast<uint32_t*>(bars + 19);
  int* s_fail = reinterpret_cast<int*>(s_taddr + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(qfull, 1);
    mbar_init(ofull, 1);
    for (int s = 0; s < kPfStages; s++) {
      mbar_init(kfull(s), 1);
      mbar_init(kempty(s), 1);
      mbar_init(vfull(s), 1);
      mbar_init(vempty(s), 1);
    }
    for (int b = 0; b < kPfSBufs; b++) {
      mbar_init(sfull(b), 1);
      mbar_init(pfull(b), 128);
      mbar_init(pvdone(b), 1);
    }
    *s_fail = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(s_taddr), kPfCols);
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
    // ---- producer: Q once, then K(j+1) ahead of V(j), the order the MMAs need them ----
    if (lane == 0) {
      mbar_expect_tx(qfull, kPfTile);
      for (int h = 0; h < 2; h++)
        tma_load_3d(smem_u32(smem + h * kPfHalf), &tq, 64 * h, hq, (int)(t0 + r0), qfull);
      int last_k[kPfStages] = {-1, -1}, last_v[kPfStages] = {-1, -1};
      auto load_k = [&](int t) {
        const int s = t & 1;
        if (t >= 2 && !mbar_wait_bounded(kempty(s), ((t >> 1) - 1) & 1)) return false;
        mbar_expect_tx(kfull(s), kPfTile);
        for (int h = 0; h < 2; h++)
          tma_load_3d(smem_u32(smem + kPfOffK + s * kPfTile + h * kPfHalf), &tk, 64 * h, kvh,
                      (int)(t0 + (long long)t * kPfT), kfull(s));
        last_k[s] = t;
        return true;
      };
      auto load_v = [&](int t) {
        const int s = t & 1;
        if (t >= 2 && !mbar_wait_bounded(vempty(s), ((t >> 1) - 1) & 1)) return false;
        mbar_expect_tx(vfull(s), kPfTile);
        for (int h = 0; h < 2; h++)
          tma_load_3d(smem_u32(smem + kPfOffV + s * kPfTile + h * kPfHalf), &tv, 64 * h, kvh,
                      (int)(t0 + (long long)t * kPfT), vfull(s));
        last_v[s] = t;
        return true;
      };
      if (!load_k(0)) fail(21);
      for (int j = 0; j < nkt && !failed(); j++) {
        if (j + 1 < nkt && !load_k(j + 1)) { fail(21); break; }
        if (!load_v(j)) { fail(22); break; }
      }
      // no copy of this CTA may still be in flight when it exits
      mbar_wait_bounded(qfull, 0);
      for (int s = 0; s < kPfStages; s++) {
        if (last_k[s] >= 0) mbar_wait_bounded(kfull(s), (last_k[s] >> 1) & 1);
        if (last_v[s] >= 0) mbar_wait_bounded(vfull(s), (last_v[s] >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: QK(0), then QK(j+1) ahead of PV(j) ----
    if (lane == 0) {
      constexpr uint32_t id_qk = umma_idesc_f16(128, 128);
      constexpr uint32_t id_pv = umma_idesc_f16(128, 128) | (1u << 16);   // B (V) MN-major
      const uint32_t qs = smem_u32(smem);
      bool ok = mbar_wait_bounded(qfull, 0);
      auto issue_qk = [&](int t) {
        const int b = t % kPfSBufs, s = t & 1;
        if (t >= kPfSBufs && !mbar_wait_bounded(pvdone(b), ((t / kPfSBufs) - 1) & 1)) return false;
        if (!mbar_wait_bounded(kfull(s), (t >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t ks = smem_u32(smem + kPfOffK + s * kPfTile);
#pragma unroll
        for (int k = 0; k < 8; k++) {
          const uint32_t off = (k >> 2) * kPfHalf + (k & 3) * 32;   // feature half, 16-feature step
          umma_f16(tbase + b * 128, umma_desc_sw128(qs + off), umma_desc_sw128(ks + off), id_qk, k > 0);
        }
        umma_commit(kempty(s));
        umma_commit(sfull(b));
        return true;
      };
      auto issue_pv = [&](int t) {
        const int b = t % kPfSBufs, s = t & 1;
        if (!mbar_wait_bounded(pfull(b), (t / kPfSBufs) & 1)) return false;
        if (!mbar_wait_bounded(vfull(s), (t >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t vs = smem_u32(smem + kPfOffV + s * kPfTile);
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {   // 16 keys a step: two 8-key groups of the V tile
          const uint64_t bd = umma_desc_sw128_mn(vs + kk * 2048, kPfHalf);
          umma_f16_tmem_a(tbase + kPfOCol, tbase + b * 128 + 8 * kk, bd, id_pv, t > 0 || kk > 0);
          umma_f16_tmem_a(tbase + kPfOCol, tbase + b * 128 + 64 + 8 * kk, bd, id_pv, true);
        }
        umma_commit(vempty(s));
        umma_commit(pvdone(b));
        return true;
      };
      if (ok && !issue_qk(0)) ok = false;
      for (int j = 0; ok && j < nkt && !failed(); j++) {
        if (j + 1 < nkt && !issue_qk(j + 1)) { ok = false; break; }
        if (!issue_pv(j)) { ok = false; break; }
      }
      if (!ok) fail(23);
      umma_commit(ofull);                     // every MMA issued so far has completed
      mbar_wait_bounded(ofull, 0);
    }
  } else {
    // ---- softmax: warps 2..5, thread = query row (lane group warp % 4) ----
    const int lg = warp & 3, row = 32 * lg + lane, prow = r0 + row;
    const uint32_t tl = tbase + ((uint32_t)(32 * lg) << 16);
    constexpr float sc = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
    float m = -INFINITY, l = 0.0f;    // base-2 maximum the probabilities are taken against, their sum
    bool ok = true;
    for (int j = 0; j < nkt; j++) {
      const int b = j % kPfSBufs;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(sfull(b), (j / kPfSBufs) & 1) && !failed());
      if (!ok) break;
      tc_fence_after();
      float x[128];
#pragma unroll
      for (int c = 0; c < 4; c++) tmem_ld32_nowait(tl + b * 128 + 32 * c, x + 32 * c);
      tmem_wait_ld();
      if (j == qt) {                   // diagonal tile: keys after the row
#pragma unroll
        for (int c = 0; c < 128; c++)
          if (j * kPfT + c > prow) x[c] = -INFINITY;
      }
      float mx = x[0];
#pragma unroll
      for (int c = 1; c < 128; c++) mx = fmaxf(mx, x[c]);
      const float mxs = mx * sc;
      // raise the row maxima of the warp when one of them would let a
      // probability exceed 2^8 (the first tile sets them)
      if (__any_sync(0xffffffffu, !(mxs <= m + kPfLazy))) {
        const float mn = fmaxf(m, mxs);
        if (j > 0) {                   // O holds tiles 0 .. j-1 against the old maxima
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(pvdone((j - 1) % kPfSBufs), ((j - 1) / kPfSBufs) & 1));
          if (!ok) break;
          tc_fence_after();
          const float f = fast_exp2(m - mn);
          l *= f;
#pragma unroll 1
          for (int c = 0; c < 4; c++) {
            float o[32];
            tmem_ld32_nowait(tl + kPfOCol + 32 * c, o);
            tmem_wait_ld();
            uint32_t w[32];
#pragma unroll
            for (int e = 0; e < 32; e++) w[e] = __float_as_uint(o[e] * f);
            tmem_st32(tl + kPfOCol + 32 * c, w);
          }
          tmem_wait_st();
        }
        m = mn;
      }
      // P over S: pair columns [0, 64), residual columns [64, 128) of the buffer
#pragma unroll
      for (int c = 0; c < 4; c++) {
        uint32_t ph[16], pr[16];
#pragma unroll
        for (int e = 0; e < 16; e++) {
          const float p0 = fast_exp2(fmaf(x[32 * c + 2 * e], sc, -m));
          const float p1 = fast_exp2(fmaf(x[32 * c + 2 * e + 1], sc, -m));
          l += p0 + p1;
          split_half2(p0, p1, ph[e], pr[e]);
        }
        tmem_st16(tl + b * 128 + 16 * c, ph);
        tmem_st16(tl + b * 128 + 64 + 16 * c, pr);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(pfull(b));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(ofull, 0) && !failed());
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      float* dst = a.out + ((t0 + prow) * Hq + hq) * kD;
#pragma unroll 1
      for (int c = 0; c < 4; c++) {
        float o[32];
        tmem_ld32_nowait(tl + kPfOCol + 32 * c, o);
        tmem_wait_ld();
        if (prow < n0) {
          float4* d4 = reinterpret_cast<float4*>(dst + 32 * c);
#pragma unroll
          for (int e = 0; e < 8; e++)
            d4[e] = make_float4(o[4 * e] * inv, o[4 * e + 1] * inv, o[4 * e + 2] * inv, o[4 * e + 3] * inv);
        }
      }
      if (a.lse_obs != nullptr) {
        float* lo = a.lse_obs + ((size_t)i * Hq + hq) * kObs;
        const int o = prow - (n0 - kObs);
        if (prow < n0 && o >= 0) lo[o] = l > 0.0f ? m + log2f(l) : -INFINITY;
        if (qt == 0 && row < kObs - n0) lo[row] = -INFINITY;   // rows before the prompt's start
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, kPfCols);
  }
}

cudaError_t configure_prefill() {
  return cudaFuncSetAttribute(k_prefill_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
}

namespace {
// [n_tok][heads][128] fp16: box = 128 rows x one head x 64 features, 128-byte swizzle
cudaError_t rows_map(PFN_cuTensorMapEncodeTiled_v12000 enc, const __half* base, int heads, long long n_tok,
                     CUtensorMap* m) {
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)heads, (cuuint64_t)n_tok};
  const cuuint64_t str[2] = {(cuuint64_t)kD * 2, (cuuint64_t)heads * kD * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)kPfT};
  const cuuint32_t es[3] = {1, 1, 1};
  if (enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half*>(base), dims, str, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_prefill(Pool& P, const CallArgs& args, int max_len, const __half* q, const __half* k,
                           const __half* v, float* out, float* lse_obs, cudaStream_t st) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  cudaError_t e = tma_encoder(&enc);
  if (e != cudaSuccess) return e;
  const long long n_tok = args.tok0[args.n_req];
  const int hkv = P.pv.hkv, hq = hkv * P.pv.G;
  CUtensorMap mq, mk, mv;
  if ((e = rows_map(enc, q, hq, n_tok, &mq)) != cudaSuccess) return e;
  if ((e = rows_map(enc, k, hkv, n_tok, &mk)) != cudaSuccess) return e;
  if ((e = rows_map(enc, v, hkv, n_tok, &mv)) != cudaSuccess) return e;
  const dim3 grid((max_len + kPfT - 1) / kPfT, hq, args.n_req);
  k_prefill_tc<<<grid, kPfThreads, kPfSmem, st>>>(P.pv, mq, mk, mv, PrefillTcArgs{out, lse_obs}, args);
  return cudaGetLastError();
}

}  // namespace dkv
