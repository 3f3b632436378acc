// attention.cu — GQA decode attention over mixed-precision unified pages
// (DiffKV, system implementation: custom attention kernel — hi pages first,
// then lo pages, sequence split with a merge; background: attention equation).
//
// Work unit: 16 consecutive slots of one tier ("chunk"). A KV head's chunk
// sequence is its hi chunks, then its lo chunks; a CTA (4 warps) takes a
// contiguous range of chunks (a split), each warp every 4th chunk.
//
// Per chunk, with G <= 8 query heads on the mma N dimension:
//   S^T[16 tok x 8 q]   = Kcodes[16 x 128] . Q^T        (m16n8k16, 8 k-steps)
//   logit = s_k (q.code) + z_k sum(q)                   (k^ = s_k code + z_k)
//   P' = p * s_v, transposed in registers (movmatrix)   (v^ = s_v code + z_v)
//   O^T[128 x 8]       += Vcodes^T[128 x 16] . P'^T      (8 m-tiles)
//   zsum[q]           += sum_tok p z_v                   (added to every feature)
// Codes become exact fp16 integers in registers (byte/nibble placed under a
// 1024 exponent, then the 1024 removed by hsub2/hfma2).
#include "dkv_kernels.cuh"

namespace dkv {

constexpr int kStages = 3;                 // cp.async ring depth per warp
constexpr int kPieces = 6;                 // 16-byte pieces per lane per chunk (hi)
constexpr int kStageBytes = kPieces * 512 + 4 * 128;

// logical row r (0..15) of a chunk -> slot offset inside the chunk; pairs
// (2t, 2t+1) and (2t+8, 2t+9) land on the 4 slots 4t..4t+3 (one value quad row,
// or two adjacent value pair rows)
__device__ __forceinline__ int chunk_slot(int r) {
  return r < 8 ? 4 * (r >> 1) + (r & 1) : 4 * ((r - 8) >> 1) + 2 + (r & 1);
}

__device__ __forceinline__ uint32_t cvt_k8(uint32_t w, uint32_t sel) {
  return hsub2_u(prmt(w, 0x64646464u, sel), 0x64006400u);
}
// 4-bit fields at bits [0,4) and [16,20) -> exact half2
__device__ __forceinline__ uint32_t cvt4_0(uint32_t w) {
  return hsub2_u(lop_and_or(w, 0x000F000Fu, 0x64006400u), 0x64006400u);
}
// 4-bit fields at bits [4,8) and [20,24)
__device__ __forceinline__ uint32_t cvt4_1(uint32_t w) {
  return hfma2_u(lop_and_or(w, 0x00F000F0u, 0x64006400u), 0x2C002C00u, 0xD400D400u);
}
// Value codes are centred before the P.V product (c - 8 for 4-bit, c - 2 for
// 2-bit; the offset goes into the zero term) so that the fp16 rounding of P'
// meets codes of both signs and largely cancels.
// 4-bit value fields at bits [0,4) / [16,20) and [4,8) / [20,24) -> c - 8
__device__ __forceinline__ uint32_t cvv4_0(uint32_t w) {
  return hsub2_u(lop_and_or(w, 0x000F000Fu, 0x64006400u), 0x64086408u);
}
__device__ __forceinline__ uint32_t cvv4_1(uint32_t w) {
  return hfma2_u(lop_and_or(w, 0x00F000F0u, 0x64006400u), 0x2C002C00u, 0xD480D480u);
}
// 2-bit value fields at bits [2b, 2b+2) and [16+2b, ...), b = 0..3 -> c - 2
__device__ __forceinline__ uint32_t cvv2_0(uint32_t w) {
  return hsub2_u(lop_and_or(w, 0x00030003u, 0x64006400u), 0x64026402u);
}
__device__ __forceinline__ uint32_t cvv2_1(uint32_t w) {
  return hfma2_u(lop_and_or(w, 0x000C000Cu, 0x64006400u), 0x34003400u, 0xDC08DC08u);
}
__device__ __forceinline__ uint32_t cvv2_2(uint32_t w) {
  return hfma2_u(lop_and_or(w, 0x00300030u, 0x64006400u), 0x2C002C00u, 0xD420D420u);
}
__device__ __forceinline__ uint32_t cvv2_3(uint32_t w) {
  return hfma2_u(lop_and_or(w, 0x00C000C0u, 0x64006400u), 0x24002400u, 0xCC80CC80u);
}

struct AttnArgs {
  const __half* q;
  float* part;        // [unit][split][G*128 + 2G]
  float* logit;       // [unit][max_chunks][16][8] (log2-domain logits)
  int cps;            // chunks per split
  int max_splits, max_chunks;
  int update;
  int layer;
};

__global__ void __launch_bounds__(128, 4) k_attn_split(PoolView pv, AttnArgs a) {
  if (pv.ctl->fail) return;
  extern __shared__ __align__(128) uint8_t smem[];
  const int split = blockIdx.x, kvh = blockIdx.y, i = blockIdx.z;
  const int slot = pv.call->slots[i];
  const int unit = i * pv.hkv + kvh;
  const int* cn = pv.cnt(a.layer, slot, kvh);
  const int nh = cn[0], nl = cn[1];
  const int ch_hi = (nh + kChunk - 1) / kChunk, ch_lo = (nl + kChunk - 1) / kChunk;
  const int total = ch_hi + ch_lo;
  const int c0 = split * a.cps;
  if (c0 >= total) return;
  const int c1 = min(total, c0 + a.cps);
  const int G = pv.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int* row = pv.row(a.layer, slot, kvh);

  // query fragments: thread (g,t) holds query g, features 32t..32t+31
  uint32_t bq_hi[8][2], bq_lo[8][2];
  float sumq_own = 0.0f;
  {
    float qf[32];
    if (g < G) {
      const uint4* qp = reinterpret_cast<const uint4*>(a.q + ((size_t)i * pv.hkv * G + (size_t)kvh * G + g) * kD + 32 * t);
#pragma unroll
      for (int x = 0; x < 4; x++) {
        const uint4 u = qp[x];
        const __half* h = reinterpret_cast<const __half*>(&u);
#pragma unroll
        for (int y = 0; y < 8; y++) qf[8 * x + y] = __half2float(h[y]);
      }
    } else {
#pragma unroll
      for (int x = 0; x < 32; x++) qf[x] = 0.0f;
    }
#pragma unroll
    for (int x = 0; x < 32; x++) sumq_own += qf[x];
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {
      bq_hi[kk][0] = pack_half2(qf[4 * kk], qf[4 * kk + 1]);
      bq_hi[kk][1] = pack_half2(qf[4 * kk + 2], qf[4 * kk + 3]);
      const int w = kk >> 1, na = (kk & 1) ? 2 : 0;
      bq_lo[kk][0] = pack_half2(qf[8 * w + na], qf[8 * w + na + 4]);
      bq_lo[kk][1] = pack_half2(qf[8 * w + na + 1], qf[8 * w + na + 5]);
    }
  }
  sumq_own += __shfl_xor_sync(0xffffffffu, sumq_own, 1);
  sumq_own += __shfl_xor_sync(0xffffffffu, sumq_own, 2);
  const float sc = 1.4426950408889634f * rsqrtf((float)kD);
  // sum(q) of the thread's two score columns (queries 2t, 2t+1), pre-scaled
  const float sq0 = __shfl_sync(0xffffffffu, sumq_own, (2 * t) * 4) * sc;
  const float sq1 = __shfl_sync(0xffffffffu, sumq_own, (2 * t + 1) * 4) * sc;

  uint8_t* wst = smem + warp * (kStages * kStageBytes);
  const int nck = (c1 - c0 - warp + 3) / 4 > 0 ? (c1 - c0 - warp + 3) / 4 : 0;   // chunks of this warp

  auto issue = [&](int x) {
    const int c = c0 + warp + 4 * x;
    uint8_t* sb = wst + (x % kStages) * kStageBytes;
    const bool hi = c < ch_hi;
    const int base = (hi ? c : c - ch_hi) * kChunk;
    const int count = hi ? nh : nl;
    const TierGeom& tg = hi ? pv.hi : pv.lo;
    const int sA = base + chunk_slot(g), sB = base + chunk_slot(g + 8);
    const bool vA = sA < count, vB = sB < count;
    const uint8_t* pA = vA ? pv.page(row[hi ? sA / tg.t : pv.L - 1 - sA / tg.t]) : pv.pages;
    const uint8_t* pB = vB ? pv.page(row[hi ? sB / tg.t : pv.L - 1 - sB / tg.t]) : pv.pages;
    const int iA = sA % tg.t, iB = sB % tg.t;
    const uint32_t s0 = smem_u32(sb) + lane * 16;
    if (hi) {
      const uint8_t* kA = pA + tg.off[0] + iA * 128 + 32 * t;
      const uint8_t* kB = pB + tg.off[0] + iB * 128 + 32 * t;
      cp_async16(s0 + 0 * 512, kA, vA ? 16 : 0);
      cp_async16(s0 + 1 * 512, kA + 16, vA ? 16 : 0);
      cp_async16(s0 + 2 * 512, kB, vB ? 16 : 0);
      cp_async16(s0 + 3 * 512, kB + 16, vB ? 16 : 0);
#pragma unroll
      for (int r2 = 0; r2 < 2; r2++) {       // value pair rows 2t and 2t+1 of the chunk
        const int s2 = base + 4 * t + 2 * r2;
        const bool vv = s2 < count;
        const uint8_t* pp = vv ? pv.page(row[s2 / tg.t]) : pv.pages;
        cp_async16(s0 + (4 + r2) * 512, pp + tg.off[1] + ((s2 % tg.t) >> 1) * 128 + 16 * g, vv ? 16 : 0);
      }
    } else {
      cp_async16(s0 + 0 * 512, pA + tg.off[0] + iA * 64 + 16 * t, vA ? 16 : 0);
      cp_async16(s0 + 1 * 512, pB + tg.off[0] + iB * 64 + 16 * t, vB ? 16 : 0);
      const int s4 = base + 4 * t;            // value quad row t of the chunk
      const bool vv = s4 < count;
      const uint8_t* pp = vv ? pv.page(row[pv.L - 1 - s4 / tg.t]) : pv.pages;
      cp_async16(s0 + 2 * 512, pp + tg.off[1] + ((s4 % tg.t) >> 2) * 128 + 16 * g, vv ? 16 : 0);
    }
    const uint32_t m0 = smem_u32(sb + kPieces * 512) + lane * 4;
    cp_async4(m0 + 0 * 128, pA + tg.off[2] + 4 * iA, vA ? 4 : 0);
    cp_async4(m0 + 1 * 128, pB + tg.off[2] + 4 * iB, vB ? 4 : 0);
    cp_async4(m0 + 2 * 128, pA + tg.off[3] + 4 * iA, vA ? 4 : 0);
    cp_async4(m0 + 3 * 128, pB + tg.off[3] + 4 * iB, vB ? 4 : 0);
  };

  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; mt++)
#pragma unroll
    for (int x = 0; x < 4; x++) o[mt][x] = 0.0f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f}, z_run[2] = {0.0f, 0.0f};

#pragma unroll
  for (int x = 0; x < kStages - 1; x++) {
    if (x < nck) issue(x);
    cp_async_commit();
  }
  for (int x = 0; x < nck; x++) {
    if (x + kStages - 1 < nck) issue(x + kStages - 1);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    const int c = c0 + warp + 4 * x;
    const bool hi = c < ch_hi;
    const int base = (hi ? c : c - ch_hi) * kChunk;
    const int count = hi ? nh : nl;
    const uint8_t* sb = wst + (x % kStages) * kStageBytes;
    const uint32_t* meta = reinterpret_cast<const uint32_t*>(sb + kPieces * 512) + lane;
    const uint32_t kmA = meta[0], kmB = meta[32], vmA = meta[64], vmB = meta[96];
    const bool vA = base + chunk_slot(g) < count, vB = base + chunk_slot(g + 8) < count;

    // ---- S^T = K . Q^T ----
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    uint4 vq0, vq1;
    if (hi) {
      const uint4 ka0 = *reinterpret_cast<const uint4*>(sb + 0 * 512 + lane * 16);
      const uint4 ka1 = *reinterpret_cast<const uint4*>(sb + 1 * 512 + lane * 16);
      const uint4 kb0 = *reinterpret_cast<const uint4*>(sb + 2 * 512 + lane * 16);
      const uint4 kb1 = *reinterpret_cast<const uint4*>(sb + 3 * 512 + lane * 16);
      vq0 = *reinterpret_cast<const uint4*>(sb + 4 * 512 + lane * 16);
      vq1 = *reinterpret_cast<const uint4*>(sb + 5 * 512 + lane * 16);
      const uint32_t kaw[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
      const uint32_t kbw[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
#pragma unroll
      for (int kk = 0; kk < 8; kk++) {
        uint32_t af[4];
        af[0] = cvt_k8(kaw[kk], 0x4140u);
        af[1] = cvt_k8(kbw[kk], 0x4140u);
        af[2] = cvt_k8(kaw[kk], 0x4342u);
        af[3] = cvt_k8(kbw[kk], 0x4342u);
        mma16816(acc, af, bq_hi[kk][0], bq_hi[kk][1]);
      }
    } else {
      const uint4 ka = *reinterpret_cast<const uint4*>(sb + 0 * 512 + lane * 16);
      const uint4 kb = *reinterpret_cast<const uint4*>(sb + 1 * 512 + lane * 16);
      vq0 = *reinterpret_cast<const uint4*>(sb + 2 * 512 + lane * 16);
      vq1 = make_uint4(0, 0, 0, 0);
      const uint32_t kaw[4] = {ka.x, ka.y, ka.z, ka.w};
      const uint32_t kbw[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
      for (int kk = 0; kk < 8; kk++) {
        const uint32_t wa = (kk & 1) ? kaw[kk >> 1] >> 8 : kaw[kk >> 1];
        const uint32_t wb = (kk & 1) ? kbw[kk >> 1] >> 8 : kbw[kk >> 1];
        uint32_t af[4];
        af[0] = cvt4_0(wa);
        af[1] = cvt4_0(wb);
        af[2] = cvt4_1(wa);
        af[3] = cvt4_1(wb);
        mma16816(acc, af, bq_lo[kk][0], bq_lo[kk][1]);
      }
    }
    // ---- logits (log2 domain), online softmax over the chunk ----
    const float skA = __half2float(__ushort_as_half((uint16_t)kmA)) , zkA = __half2float(__ushort_as_half((uint16_t)(kmA >> 16)));
    const float skB = __half2float(__ushort_as_half((uint16_t)kmB)), zkB = __half2float(__ushort_as_half((uint16_t)(kmB >> 16)));
    float l2[4];
    l2[0] = vA ? __fmaf_rn(acc[0], skA * sc, zkA * sq0) : -INFINITY;
    l2[1] = vA ? __fmaf_rn(acc[1], skA * sc, zkA * sq1) : -INFINITY;
    l2[2] = vB ? __fmaf_rn(acc[2], skB * sc, zkB * sq0) : -INFINITY;
    l2[3] = vB ? __fmaf_rn(acc[3], skB * sc, zkB * sq1) : -INFINITY;
    if (a.update && 2 * t < G) {
      float* lg = a.logit + ((size_t)unit * a.max_chunks + c) * (kChunk * 8);
      *reinterpret_cast<float2*>(lg + g * 8 + 2 * t) = make_float2(l2[0], l2[1]);
      *reinterpret_cast<float2*>(lg + (g + 8) * 8 + 2 * t) = make_float2(l2[2], l2[3]);
    }
    float cm0 = fmaxf(l2[0], l2[2]), cm1 = fmaxf(l2[1], l2[3]);
#pragma unroll
    for (int s = 4; s <= 16; s <<= 1) {
      cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, s));
      cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, s));
    }
    const float mn0 = fmaxf(m_run[0], cm0), mn1 = fmaxf(m_run[1], cm1);
    // a query column with no valid token so far keeps m = -inf and contributes nothing
    const float f0 = mn0 == -INFINITY ? 1.0f : fast_exp2(m_run[0] - mn0);
    const float f1 = mn1 == -INFINITY ? 1.0f : fast_exp2(m_run[1] - mn1);
    const float p0 = mn0 == -INFINITY ? 0.0f : fast_exp2(l2[0] - mn0);
    const float p1 = mn1 == -INFINITY ? 0.0f : fast_exp2(l2[1] - mn1);
    const float p2 = mn0 == -INFINITY ? 0.0f : fast_exp2(l2[2] - mn0);
    const float p3 = mn1 == -INFINITY ? 0.0f : fast_exp2(l2[3] - mn1);
    m_run[0] = mn0; m_run[1] = mn1;
    // v^ = s (c - off) + (z + off s), off = 8 (hi) or 2 (lo)
    const float voff = hi ? 8.0f : 2.0f;
    const float svA = vA ? __half2float(__ushort_as_half((uint16_t)vmA)) : 0.0f;
    const float zvA = vA ? __fmaf_rn(voff, svA, __half2float(__ushort_as_half((uint16_t)(vmA >> 16)))) : 0.0f;
    const float svB = vB ? __half2float(__ushort_as_half((uint16_t)vmB)) : 0.0f;
    const float zvB = vB ? __fmaf_rn(voff, svB, __half2float(__ushort_as_half((uint16_t)(vmB >> 16)))) : 0.0f;
    l_run[0] = l_run[0] * f0 + p0 + p2;
    l_run[1] = l_run[1] * f1 + p1 + p3;
    z_run[0] = z_run[0] * f0 + p0 * zvA + p2 * zvB;
    z_run[1] = z_run[1] * f1 + p1 * zvA + p3 * zvB;
#pragma unroll
    for (int mt = 0; mt < 8; mt++) {
      o[mt][0] *= f0; o[mt][2] *= f0;
      o[mt][1] *= f1; o[mt][3] *= f1;
    }
    // P'^T as B fragments: block of tokens 0-7 and block of tokens 8-15
    const uint32_t pb0 = movmatrix_trans(pack_half2(p0 * svA, p1 * svA));
    const uint32_t pb1 = movmatrix_trans(pack_half2(p2 * svB, p3 * svB));
    // ---- O^T += V^T . P'^T ----
    const uint32_t vw0[4] = {vq0.x, vq0.y, vq0.z, vq0.w};
    const uint32_t vw1[4] = {vq1.x, vq1.y, vq1.z, vq1.w};
    if (hi) {
#pragma unroll
      for (int mt = 0; mt < 8; mt++) {
        const uint32_t w0 = (mt & 1) ? vw0[mt >> 1] >> 8 : vw0[mt >> 1];
        const uint32_t w1 = (mt & 1) ? vw1[mt >> 1] >> 8 : vw1[mt >> 1];
        uint32_t af[4];
        af[0] = cvv4_0(w0);   // feature 16g+2mt,   tokens 2t,2t+1
        af[1] = cvv4_1(w0);   // feature 16g+2mt+1, tokens 2t,2t+1
        af[2] = cvv4_0(w1);   // feature 16g+2mt,   tokens 2t+8,2t+9
        af[3] = cvv4_1(w1);   // feature 16g+2mt+1, tokens 2t+8,2t+9
        mma16816(o[mt], af, pb0, pb1);
      }
    } else {
#pragma unroll
      for (int mt = 0; mt < 8; mt++) {
        const uint32_t w = (mt & 1) ? vw0[mt >> 1] >> 8 : vw0[mt >> 1];
        uint32_t af[4];
        af[0] = cvv2_0(w);    // feature 16g+2mt,   slots e0,e1
        af[1] = cvv2_2(w);    // feature 16g+2mt+1, slots e0,e1
        af[2] = cvv2_1(w);    // feature 16g+2mt,   slots e2,e3
        af[3] = cvv2_3(w);    // feature 16g+2mt+1, slots e2,e3
        mma16816(o[mt], af, pb0, pb1);
      }
    }
  }
  cp_async_wait<0>();
  // ---- reduce the warp's state and merge the 4 warps ----
#pragma unroll
  for (int s = 4; s <= 16; s <<= 1) {
    l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], s);
    l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], s);
    z_run[0] += __shfl_xor_sync(0xffffffffu, z_run[0], s);
    z_run[1] += __shfl_xor_sync(0xffffffffu, z_run[1], s);
  }
  __syncthreads();   // every warp is done with its stages; reuse them
  float* sO = reinterpret_cast<float*>(smem);            // [warp][8 q][128 f]
  float* sM = sO + kAttnWarps * 8 * kD;                  // [warp][8] m, l, z
  float* sL = sM + kAttnWarps * 8;
  float* sZ = sL + kAttnWarps * 8;
#pragma unroll
  for (int mt = 0; mt < 8; mt++) {
    const int f = 16 * g + 2 * mt;
    sO[(warp * 8 + 2 * t) * kD + f] = o[mt][0];
    sO[(warp * 8 + 2 * t + 1) * kD + f] = o[mt][1];
    sO[(warp * 8 + 2 * t) * kD + f + 1] = o[mt][2];
    sO[(warp * 8 + 2 * t + 1) * kD + f + 1] = o[mt][3];
  }
  if (g == 0) {
    sM[warp * 8 + 2 * t] = m_run[0]; sM[warp * 8 + 2 * t + 1] = m_run[1];
    sL[warp * 8 + 2 * t] = l_run[0]; sL[warp * 8 + 2 * t + 1] = l_run[1];
    sZ[warp * 8 + 2 * t] = z_run[0]; sZ[warp * 8 + 2 * t + 1] = z_run[1];
  }
  __syncthreads();
  float* dst = a.part + ((size_t)unit * a.max_splits + split) * (G * (kD + 2));
  for (int idx = threadIdx.x; idx < G * kD; idx += blockDim.x) {
    const int qh = idx / kD, f = idx % kD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; w++) M = fmaxf(M, sM[w * 8 + qh]);
    float O = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kAttnWarps; w++) {
        const float mw = sM[w * 8 + qh];
        if (mw != -INFINITY) O += fast_exp2(mw - M) * (sO[(w * 8 + qh) * kD + f] + sZ[w * 8 + qh]);
      }
    }
    dst[qh * kD + f] = O;
  }
  if (threadIdx.x < G) {
    const int qh = threadIdx.x;
    float M = -INFINITY, L = 0.0f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; w++) M = fmaxf(M, sM[w * 8 + qh]);
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kAttnWarps; w++) {
        const float mw = sM[w * 8 + qh];
        if (mw != -INFINITY) L += fast_exp2(mw - M) * sL[w * 8 + qh];
      }
    }
    dst[G * kD + qh] = M;
    dst[G * kD + G + qh] = L;
  }
}

// Merge the splits of each (request, KV head): out = sum_s 2^(m_s-M) O_s /
// sum_s 2^(m_s-M) l_s; lse2 = M + log2(L) (log2 domain) for the score update.
__global__ void __launch_bounds__(128) k_attn_merge(PoolView pv, AttnArgs a, float* out, float* lse2) {
  if (pv.ctl->fail) return;
  const int unit = blockIdx.x, i = unit / pv.hkv, kvh = unit % pv.hkv;
  const int slot = pv.call->slots[i];
  const int G = pv.G;
  const int* cn = pv.cnt(a.layer, slot, kvh);
  const int total = (cn[0] + kChunk - 1) / kChunk + (cn[1] + kChunk - 1) / kChunk;
  const int ns = (total + a.cps - 1) / a.cps;
  const float* src = a.part + (size_t)unit * a.max_splits * (G * (kD + 2));
  const int stride = G * (kD + 2);
  for (int idx = threadIdx.x; idx < G * kD; idx += blockDim.x) {
    const int qh = idx / kD, f = idx % kD;
    float M = -INFINITY;
    for (int s = 0; s < ns; s++) M = fmaxf(M, src[s * stride + G * kD + qh]);
    float O = 0.0f, L = 0.0f;
    if (M != -INFINITY) {
      for (int s = 0; s < ns; s++) {
        const float ms = src[s * stride + G * kD + qh];
        if (ms == -INFINITY) continue;
        const float w = exp2f(ms - M);
        O += w * src[s * stride + qh * kD + f];
        L += w * src[s * stride + G * kD + G + qh];
      }
    }
    out[((size_t)i * pv.hkv * G + (size_t)kvh * G + qh) * kD + f] = L > 0.0f ? O / L : 0.0f;
    if (f == 0) lse2[(size_t)unit * G + qh] = L > 0.0f ? M + log2f(L) : -INFINITY;
  }
  if (a.update && kvh == 0 && threadIdx.x == 0) pv.rq(a.layer, slot)[3] += 1;
}

// Score update: every stored token's score gains max over the group's heads
// of its softmax probability, 2^(l2 - lse2).
__global__ void __launch_bounds__(256) k_attn_scores(PoolView pv, AttnArgs a, const float* __restrict__ lse2) {
  if (pv.ctl->fail) return;
  const int unit = blockIdx.y, i = unit / pv.hkv, kvh = unit % pv.hkv;
  const int slot = pv.call->slots[i];
  const int G = pv.G;
  const int* cn = pv.cnt(a.layer, slot, kvh);
  const int nh = cn[0], nl = cn[1];
  const int ch_hi = (nh + kChunk - 1) / kChunk;
  const int c = blockIdx.x * (blockDim.x / kChunk) + threadIdx.x / kChunk;
  const int r = threadIdx.x % kChunk;
  const int total = ch_hi + (nl + kChunk - 1) / kChunk;
  if (c >= total) return;
  const bool hi = c < ch_hi;
  const int s = (hi ? c : c - ch_hi) * kChunk + chunk_slot(r);
  if (s >= (hi ? nh : nl)) return;
  const float* lg = a.logit + ((size_t)unit * a.max_chunks + c) * (kChunk * 8) + r * 8;
  float pm = 0.0f;
  for (int qh = 0; qh < G; qh++) pm = fmaxf(pm, exp2f(lg[qh] - lse2[(size_t)unit * G + qh]));
  const int* row = pv.row(a.layer, slot, kvh);
  const TierGeom& tg = hi ? pv.hi : pv.lo;
  uint8_t* pg = pv.page(row[hi ? s / tg.t : pv.L - 1 - s / tg.t]);
  float* sp = reinterpret_cast<float*>(pg + tg.off[4] + 4 * (s % tg.t));
  *sp = *sp + pm;
}

int attn_smem_bytes() {
  const int ring = kAttnWarps * kStages * kStageBytes;
  const int merge = (kAttnWarps * 8 * kD + 3 * kAttnWarps * 8) * 4;
  return ring > merge ? ring : merge;
}

cudaError_t launch_attention(Pool& P, int layer, int n_req, int max_tokens, const __half* q, float* out,
                             int update_scores, cudaStream_t st) {
  AttnArgs a;
  a.q = q;
  a.part = P.sc.apart;
  a.logit = P.sc.alogit;
  a.max_splits = P.sc.max_splits;
  a.max_chunks = P.sc.max_chunks;
  a.update = update_scores;
  a.layer = layer;
  const int max_chunks_call = (max_tokens + kChunk - 1) / kChunk + 1;
  // split length: enough CTAs for several waves, at least 8 chunks per split
  const long long units = (long long)n_req * P.pv.hkv;
  int cps = (int)((units * max_chunks_call + 152LL * 24 - 1) / (152LL * 24));
  cps = cps < 8 ? 8 : cps;
  cps = (cps + 3) / 4 * 4;
  int ns = (max_chunks_call + cps - 1) / cps;
  if (ns > P.sc.max_splits) {
    ns = P.sc.max_splits;
    cps = (max_chunks_call + ns - 1) / ns;
  }
  a.cps = cps;
  const dim3 grid(ns, P.pv.hkv, n_req);
  k_attn_split<<<grid, 128, attn_smem_bytes(), st>>>(P.pv, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_attn_merge<<<(unsigned)units, 128, 0, st>>>(P.pv, a, out, P.sc.alse);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (update_scores) {
    const dim3 g2((max_chunks_call + 15) / 16, (unsigned)units);
    k_attn_scores<<<g2, 256, 0, st>>>(P.pv, a, P.sc.alse);
    e = cudaGetLastError();
  }
  return e;
}

cudaError_t configure_attention() {
  return cudaFuncSetAttribute(k_attn_split, cudaFuncAttributeMaxDynamicSharedMemorySize, attn_smem_bytes());
}

}  // namespace dkv
