// prefill.cu — causal GQA attention over the prompt, the model's own
// attention that DiffKV's compactor follows (DiffKV, system implementation:
// the compactor runs after the attention of each layer; background: the
// attention equation). Its last 32 query rows also leave their base-2
// log-sum-exps, which the prompt score pass takes in place of its own pass
// over the keys (dkv_compact_step_prefilled).
//
// One CTA per (64 query rows, query head, request), 4 warps of 16 rows. Key
// and value tiles of 64 rows are staged in shared memory by cp.async (two
// stages, 16-byte chunks XOR-swizzled by row so that ldmatrix's eight rows
// fall in different banks); per tile each warp computes S = Q K^T
// (m16n8k16, fp32 accumulators), keeps an online softmax in base 2 and adds
// P V, P entering as an fp16 pair plus its fp16 residual (about 22
// significant bits, so that the element-wise bound holds next to outlier
// channels). Query tiles are taken heaviest (longest causal range) first.
#include <algorithm>

#include "dkv_kernels.cuh"

namespace dkv {

constexpr int kPfRows = 64;                      // query rows per CTA
constexpr int kPfKeys = 64;                      // keys per staged tile
constexpr int kPfWarps = 4;
constexpr int kPfTileBytes = kPfKeys * kD * 2;   // one K or V tile, 16 KB
constexpr int kPfSmem = 2 * 2 * kPfTileBytes;    // two stages of K and V

struct PrefillArgs {
  const __half* q;     // [tokens][Hq][128]
  const __half* k;     // [tokens][Hkv][128]
  const __half* v;
  float* out;          // [tokens][Hq][128]
  float* lse_obs;      // [n_req][Hq][32] or null
};

// byte offset of 16-byte chunk c of row r in a staged tile (256-byte rows)
__device__ __forceinline__ uint32_t pf_off(int r, int c) { return (uint32_t)(r * 256 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__global__ void __launch_bounds__(32 * kPfWarps) k_prefill(PoolView pv, PrefillArgs a, const __grid_constant__ CallArgs ca) {
  if (pv.noop()) return;
  extern __shared__ __align__(128) uint8_t smem[];
  const int hq = blockIdx.y, i = blockIdx.z;
  const int G = pv.G, Hq = pv.hkv * G, kvh = hq / G;
  const int n0 = ca.lens[i];
  const int ntiles = (n0 + kPfRows - 1) / kPfRows;
  if ((int)blockIdx.x >= ntiles) return;
  const int qt = ntiles - 1 - (int)blockIdx.x;   // heaviest tiles first
  const int r0 = qt * kPfRows;
  const long long t0 = ca.tok0[i];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int rowA = r0 + 16 * warp + g, rowB = rowA + 8;   // the thread's two rows
  // Q fragments of the warp's 16 rows: 8 k-steps of 16 features
  uint32_t qa[8][4];
  {
    const uint32_t* qA = reinterpret_cast<const uint32_t*>(a.q + ((t0 + rowA) * Hq + hq) * kD);
    const uint32_t* qB = reinterpret_cast<const uint32_t*>(a.q + ((t0 + rowB) * Hq + hq) * kD);
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {
      qa[kk][0] = rowA < n0 ? __ldg(qA + kk * 8 + t) : 0u;
      qa[kk][1] = rowB < n0 ? __ldg(qB + kk * 8 + t) : 0u;
      qa[kk][2] = rowA < n0 ? __ldg(qA + kk * 8 + 4 + t) : 0u;
      qa[kk][3] = rowB < n0 ? __ldg(qB + kk * 8 + 4 + t) : 0u;
    }
  }
  // key tile kt into stage s (K then V), keys past the prompt zero-filled
  auto stage = [&](int kt, int s) {
    uint8_t* ks = smem + s * 2 * kPfTileBytes;
    uint8_t* vs = ks + kPfTileBytes;
    for (int x = threadIdx.x; x < kPfKeys * 16; x += blockDim.x) {
      const int r = x >> 4, c = x & 15;
      const int j = kt * kPfKeys + r;
      const bool ok = j < n0;
      const size_t row = ((size_t)(t0 + (ok ? j : 0)) * pv.hkv + kvh) * kD + 8 * c;
      cp_async16(smem_u32(ks + pf_off(r, c)), a.k + row, ok ? 16 : 0);
      cp_async16(smem_u32(vs + pf_off(r, c)), a.v + row, ok ? 16 : 0);
    }
    cp_async_commit();
  };
  const int nkt = qt + 1;         // key tiles 0 .. qt hold every key at or before the tile's rows
  stage(0, 0);
  constexpr float sc = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
  float o[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; nt++) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.0f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;   // rows A and B (this thread's columns)
  for (int kt = 0; kt < nkt; kt++) {
    if (kt + 1 < nkt) {
      stage(kt + 1, (kt + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t ks = smem_u32(smem + (kt & 1) * 2 * kPfTileBytes), vs = ks + kPfTileBytes;
    // S = Q K^T over 8 n-tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; nt++) {
      s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.0f;
#pragma unroll
      for (int k2 = 0; k2 < 4; k2++) {   // two k-steps per ldmatrix
        uint32_t b[4];
        ldmatrix_x4(b, ks + pf_off(nt * 8 + (lane & 7), 4 * k2 + (lane >> 3)));
        mma16816(s[nt], qa[2 * k2], b[0], b[1]);
        mma16816(s[nt], qa[2 * k2 + 1], b[2], b[3]);
      }
    }
    // scale to base 2; on the diagonal tile mask keys after the row (and past the prompt)
#pragma unroll
    for (int nt = 0; nt < 8; nt++)
#pragma unroll
      for (int e = 0; e < 4; e++) {
        float x = s[nt][e] * sc;
        if (kt == qt) {
          const int j = kt * kPfKeys + nt * 8 + 2 * t + (e & 1);
          const int row = e < 2 ? rowA : rowB;
          if (j > row || j >= n0) x = -INFINITY;
        }
        s[nt][e] = x;
      }
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; nt++) {
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
#pragma unroll
    for (int sh = 1; sh <= 2; sh <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float b0 = mn0 == -INFINITY ? 0.0f : mn0, b1 = mn1 == -INFINITY ? 0.0f : mn1;   // rows with no key yet
    const float f0 = fast_exp2(m0 - b0), f1 = fast_exp2(m1 - b1);
    m0 = mn0;
    m1 = mn1;
    l0 *= f0;
    l1 *= f1;
#pragma unroll
    for (int nt = 0; nt < 16; nt++) {
      o[nt][0] *= f0;
      o[nt][1] *= f0;
      o[nt][2] *= f1;
      o[nt][3] *= f1;
    }
#pragma unroll
    for (int nt = 0; nt < 8; nt++) {
      s[nt][0] = fast_exp2(s[nt][0] - b0);
      s[nt][1] = fast_exp2(s[nt][1] - b0);
      s[nt][2] = fast_exp2(s[nt][2] - b1);
      s[nt][3] = fast_exp2(s[nt][3] - b1);
      l0 += s[nt][0] + s[nt][1];
      l1 += s[nt][2] + s[nt][3];
    }
    // O += P V: 4 k-steps of 16 keys, P as an fp16 pair plus its residual
#pragma unroll
    for (int kk = 0; kk < 4; kk++) {
      uint32_t ph[4], pr[4];
      split_half2(s[2 * kk][0], s[2 * kk][1], ph[0], pr[0]);
      split_half2(s[2 * kk][2], s[2 * kk][3], ph[1], pr[1]);
      split_half2(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[2], pr[2]);
      split_half2(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[3], pr[3]);
#pragma unroll
      for (int dn = 0; dn < 8; dn++) {   // pairs of 8-feature n-tiles
        uint32_t b[4];
        ldmatrix_x4_trans(b, vs + pf_off(kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, 2 * dn + (lane >> 4)));
        mma16816(o[2 * dn], ph, b[0], b[1]);
        mma16816(o[2 * dn], pr, b[0], b[1]);
        mma16816(o[2 * dn + 1], ph, b[2], b[3]);
        mma16816(o[2 * dn + 1], pr, b[2], b[3]);
      }
    }
    __syncthreads();              // every warp is done with this stage before it is refilled
  }
#pragma unroll
  for (int sh = 1; sh <= 2; sh <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, sh);
    l1 += __shfl_xor_sync(0xffffffffu, l1, sh);
  }
  const float inv0 = l0 > 0.0f ? 1.0f / l0 : 0.0f, inv1 = l1 > 0.0f ? 1.0f / l1 : 0.0f;
  if (rowA < n0) {
    float* dst = a.out + ((t0 + rowA) * Hq + hq) * kD + 2 * t;
#pragma unroll
    for (int nt = 0; nt < 16; nt++)
      *reinterpret_cast<float2*>(dst + nt * 8) = make_float2(o[nt][0] * inv0, o[nt][1] * inv0);
  }
  if (rowB < n0) {
    float* dst = a.out + ((t0 + rowB) * Hq + hq) * kD + 2 * t;
#pragma unroll
    for (int nt = 0; nt < 16; nt++)
      *reinterpret_cast<float2*>(dst + nt * 8) = make_float2(o[nt][2] * inv1, o[nt][3] * inv1);
  }
  if (a.lse_obs != nullptr) {
    float* lo = a.lse_obs + ((size_t)i * Hq + hq) * kObs;
    if (t == 0) {                 // observation rows: positions n0 - 32 .. n0 - 1
      const int oa = rowA - (n0 - kObs), ob = rowB - (n0 - kObs);
      if (rowA < n0 && oa >= 0) lo[oa] = l0 > 0.0f ? m0 + log2f(l0) : -INFINITY;
      if (rowB < n0 && ob >= 0) lo[ob] = l1 > 0.0f ? m1 + log2f(l1) : -INFINITY;
    }
    if (qt == 0)                  // rows of negative positions (prompts shorter than 32)
      for (int x = threadIdx.x; x < kObs - n0; x += blockDim.x) lo[x] = -INFINITY;
  }
}

cudaError_t configure_prefill() {
  return cudaFuncSetAttribute(k_prefill, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
}

cudaError_t launch_prefill(Pool& P, const CallArgs& args, int max_len, const __half* q, const __half* k,
                           const __half* v, float* out, float* lse_obs, cudaStream_t st) {
  PrefillArgs a{q, k, v, out, lse_obs};
  const dim3 grid((max_len + kPfRows - 1) / kPfRows, P.pv.hkv * P.pv.G, args.n_req);
  k_prefill<<<grid, 32 * kPfWarps, kPfSmem, st>>>(P.pv, a, args);
  return cudaGetLastError();
}

}  // namespace dkv
