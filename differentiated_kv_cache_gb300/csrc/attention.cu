// attention.cu — GQA decode attention over mixed-precision unified pages
// (DiffKV, system implementation: custom attention kernel — hi pages first,
// then lo pages, sequence split with a merge; background: attention equation).
//
// Work unit: 16 consecutive slots of one tier ("chunk"). Per chunk, with
// G <= 8 query heads on the mma N dimension:
//   S^T[16 tok x 8 q]   = Kcodes[16 x 128] . Q^T        (m16n8k16, 8 k-steps)
//   logit = s_k (q.code) + z_k sum(q)                   (k^ = s_k code + z_k)
//   P' = p * s_v, transposed in registers (movmatrix)   (v^ = s_v code + z_v)
//   O^T[128 x 8]       += Vcodes^T[128 x 16] . P'^T      (8 m-tiles)
//   zsum[q]           += sum_tok p z_v                   (added to every feature)
// Codes become exact fp16 integers in registers (byte/nibble placed under a
// 1024 exponent, then the 1024 removed by hsub2/hfma2).
//
// Work distribution: the sequences of all KV heads of the call are
// concatenated and cut into equal contiguous ranges, one per warp of a
// persistent grid (the sequence split of the page's kernel, balanced). A warp
// writes a partial (m, l, O) for every head its range touches; the last warp
// to finish a head merges the head's partials. Data is staged in shared memory
// by bulk asynchronous copies completing on per-stage mbarriers:
//   k_attn_paged   pages of 16k tokens (chunk-aligned): one copy per page of
//                  its contiguous K | V | K-meta | V-meta prefix;
//   k_attn_decode  any page geometry: per 16-slot chunk, one copy per page run.
#include <algorithm>
#include <mutex>

#include "dkv_kernels.cuh"

namespace dkv {

constexpr int kStages = 3;                 // ring depth per warp (chunked path)
constexpr int kPageStages = 4;             // ring depth per warp (paged path)
constexpr int kMinChunks = 8;              // ring work items per warp at least
constexpr int kCtasPerSm = 3;
constexpr int kOffV = 2048;                // chunked stage image: V rows
constexpr int kOffMeta = 3072;             // chunked stage image: page meta segments

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

__host__ __device__ constexpr int part_stride(int G) { return G * kD + 2 * kMaxG; }

struct AttnArgs {
  const __half* q;
  float* out;         // [n_req][Hkv*G][128]
  float* part;        // [unit][max_parts][G*128 + 16]: O (G x 128), m (8), l (8); a
                      // multiple of 4 floats so every record is 16-byte aligned
  float* logit;       // [unit][max_chunks][16][8] (log2-domain logits)
  float* lse2;        // [unit][G]
  int* done;          // [unit] partials published (zero between calls)
  int max_parts, max_chunks;
  int update;
  int layer;
  int mseg;           // chunked: bytes per page meta segment in the stage
  int maxp;           // chunked: pages a chunk can touch
  int stage_bytes;
};

// A warp's position in the concatenated work sequence: the head (unit) that
// holds global item indices [begin, end); items are chunks or pages.
struct Cursor {
  int u, begin, end, nh, nl, hi_items;
  const int* row;
};

__device__ __forceinline__ void cursor_at(Cursor& c, int u, const int* s_pref, const PoolView& pv,
                                          const SlotArgs& sa, int layer, bool paged) {
  c.u = u;
  c.begin = s_pref[u];
  c.end = s_pref[u + 1];
  const int slot = sa.slots[u / pv.hkv], kvh = u % pv.hkv;
  const int* cn = pv.cnt(layer, slot, kvh);
  c.nh = cn[0];
  c.nl = cn[1];
  c.hi_items = paged ? (c.nh + pv.hi.t - 1) / pv.hi.t : (c.nh + kChunk - 1) / kChunk;
  c.row = pv.row(layer, slot, kvh);
}

__device__ __forceinline__ void cursor_seek(Cursor& c, int x, const int* s_pref, const PoolView& pv,
                                            const SlotArgs& sa, int layer, bool paged) {
  while (x >= c.end) cursor_at(c, c.u + 1, s_pref, pv, sa, layer, paged);
}

// Query fragments of one head's G query heads for thread (g,t): query g,
// features 32t..32t+31, in the feature orders of the 8-bit and 4-bit key rows.
__device__ __forceinline__ void load_q(const PoolView& pv, const AttnArgs& a, int i, int kvh, int g, int t,
                                       uint32_t (&bq_hi)[8][2], uint32_t (&bq_lo)[8][2], float& sq0, float& sq1) {
  const int G = pv.G;
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
  float sum = 0.0f;
#pragma unroll
  for (int x = 0; x < 32; x++) sum += qf[x];
#pragma unroll
  for (int kk = 0; kk < 8; kk++) {
    bq_hi[kk][0] = pack_half2(qf[4 * kk], qf[4 * kk + 1]);
    bq_hi[kk][1] = pack_half2(qf[4 * kk + 2], qf[4 * kk + 3]);
    const int w = kk >> 1, na = (kk & 1) ? 2 : 0;
    bq_lo[kk][0] = pack_half2(qf[8 * w + na], qf[8 * w + na + 4]);
    bq_lo[kk][1] = pack_half2(qf[8 * w + na + 1], qf[8 * w + na + 5]);
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  const float sc = 1.4426950408889634f * rsqrtf((float)kD);
  // sum(q) of the thread's two score columns (queries 2t, 2t+1), pre-scaled
  sq0 = __shfl_sync(0xffffffffu, sum, (2 * t) * 4) * sc;
  sq1 = __shfl_sync(0xffffffffu, sum, (2 * t + 1) * 4) * sc;
}

// Online-softmax state of one warp for one head: O^T fragments (features
// 16g+2mt(+1), queries 2t, 2t+1), running max, sum and value-zero sum.
struct AttnState {
  float o[8][4];
  float m[2], l[2], z[2];
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int mt = 0; mt < 8; mt++)
#pragma unroll
      for (int x = 0; x < 4; x++) o[mt][x] = 0.0f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.0f;
    z[0] = z[1] = 0.0f;
  }
};

// One 16-slot chunk for thread (g,t). kA/kB: key rows of tokens A (logical
// row g) and B (row g+8), at the thread's feature bytes; v0/v1: value rows at
// the thread's 16 features (hi: pair rows 2t and 2t+1; lo: quad row t in v0);
// km*/vm*: {fp16 scale, fp16 zero} of A and B; lg: logit row of the chunk or
// nullptr.
__device__ __forceinline__ void attend_chunk(AttnState& S, bool hi, const uint8_t* kA, const uint8_t* kB,
                                             const uint8_t* v0, const uint8_t* v1, uint32_t kmA, uint32_t kmB,
                                             uint32_t vmA, uint32_t vmB, bool vA, bool vB,
                                             const uint32_t (&bq_hi)[8][2], const uint32_t (&bq_lo)[8][2],
                                             float sq0, float sq1, float* lg, int G, int g, int t) {
  // ---- S^T = K . Q^T (two independent accumulator chains) ----
  float acc0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, acc1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  uint4 vq0, vq1;
  if (hi) {
    const uint4 ka0 = reinterpret_cast<const uint4*>(kA)[0], ka1 = reinterpret_cast<const uint4*>(kA)[1];
    const uint4 kb0 = reinterpret_cast<const uint4*>(kB)[0], kb1 = reinterpret_cast<const uint4*>(kB)[1];
    vq0 = *reinterpret_cast<const uint4*>(v0);
    vq1 = *reinterpret_cast<const uint4*>(v1);
    const uint32_t kaw[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
    const uint32_t kbw[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {
      uint32_t af[4];
      af[0] = cvt_k8(kaw[kk], 0x4140u);
      af[1] = cvt_k8(kbw[kk], 0x4140u);
      af[2] = cvt_k8(kaw[kk], 0x4342u);
      af[3] = cvt_k8(kbw[kk], 0x4342u);
      mma16816((kk & 1) ? acc1 : acc0, af, bq_hi[kk][0], bq_hi[kk][1]);
    }
  } else {
    const uint4 ka = *reinterpret_cast<const uint4*>(kA);
    const uint4 kb = *reinterpret_cast<const uint4*>(kB);
    vq0 = *reinterpret_cast<const uint4*>(v0);
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
      mma16816((kk & 1) ? acc1 : acc0, af, bq_lo[kk][0], bq_lo[kk][1]);
    }
  }
  // ---- logits (log2 domain), online softmax over the chunk ----
  const float sc = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
  const float skA = __half2float(__ushort_as_half((uint16_t)kmA)), zkA = __half2float(__ushort_as_half((uint16_t)(kmA >> 16)));
  const float skB = __half2float(__ushort_as_half((uint16_t)kmB)), zkB = __half2float(__ushort_as_half((uint16_t)(kmB >> 16)));
  float l2[4];
  l2[0] = vA ? __fmaf_rn(acc0[0] + acc1[0], skA * sc, zkA * sq0) : -INFINITY;
  l2[1] = vA ? __fmaf_rn(acc0[1] + acc1[1], skA * sc, zkA * sq1) : -INFINITY;
  l2[2] = vB ? __fmaf_rn(acc0[2] + acc1[2], skB * sc, zkB * sq0) : -INFINITY;
  l2[3] = vB ? __fmaf_rn(acc0[3] + acc1[3], skB * sc, zkB * sq1) : -INFINITY;
  if (lg != nullptr && 2 * t < G) {
    *reinterpret_cast<float2*>(lg + g * 8 + 2 * t) = make_float2(l2[0], l2[1]);
    *reinterpret_cast<float2*>(lg + (g + 8) * 8 + 2 * t) = make_float2(l2[2], l2[3]);
  }
  float cm0 = fmaxf(l2[0], l2[2]), cm1 = fmaxf(l2[1], l2[3]);
#pragma unroll
  for (int s = 4; s <= 16; s <<= 1) {
    cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, s));
    cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, s));
  }
  const float mn0 = fmaxf(S.m[0], cm0), mn1 = fmaxf(S.m[1], cm1);
  // a query column with no valid token so far keeps m = -inf and contributes nothing
  const float f0 = mn0 == -INFINITY ? 1.0f : fast_exp2(S.m[0] - mn0);
  const float f1 = mn1 == -INFINITY ? 1.0f : fast_exp2(S.m[1] - mn1);
  const float p0 = mn0 == -INFINITY ? 0.0f : fast_exp2(l2[0] - mn0);
  const float p1 = mn1 == -INFINITY ? 0.0f : fast_exp2(l2[1] - mn1);
  const float p2 = mn0 == -INFINITY ? 0.0f : fast_exp2(l2[2] - mn0);
  const float p3 = mn1 == -INFINITY ? 0.0f : fast_exp2(l2[3] - mn1);
  S.m[0] = mn0;
  S.m[1] = mn1;
  // v^ = s (c - off) + (z + off s), off = 8 (hi) or 2 (lo)
  const float voff = hi ? 8.0f : 2.0f;
  const float svA = vA ? __half2float(__ushort_as_half((uint16_t)vmA)) : 0.0f;
  const float zvA = vA ? __fmaf_rn(voff, svA, __half2float(__ushort_as_half((uint16_t)(vmA >> 16)))) : 0.0f;
  const float svB = vB ? __half2float(__ushort_as_half((uint16_t)vmB)) : 0.0f;
  const float zvB = vB ? __fmaf_rn(voff, svB, __half2float(__ushort_as_half((uint16_t)(vmB >> 16)))) : 0.0f;
  S.l[0] = S.l[0] * f0 + p0 + p2;
  S.l[1] = S.l[1] * f1 + p1 + p3;
  S.z[0] = S.z[0] * f0 + p0 * zvA + p2 * zvB;
  S.z[1] = S.z[1] * f1 + p1 * zvA + p3 * zvB;
  if (!__all_sync(0xffffffffu, f0 == 1.0f && f1 == 1.0f)) {
#pragma unroll
    for (int mt = 0; mt < 8; mt++) {
      S.o[mt][0] *= f0; S.o[mt][2] *= f0;
      S.o[mt][1] *= f1; S.o[mt][3] *= f1;
    }
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
      mma16816(S.o[mt], af, pb0, pb1);
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
      mma16816(S.o[mt], af, pb0, pb1);
    }
  }
}

// Publish the warp's partial of head u (items [begin, end), warp ranges of C
// items); the last warp of the head merges every partial into out and lse2.
__device__ void publish(const PoolView& pv, const AttnArgs& a, const SlotArgs& sa, AttnState& S, int u, int first,
                        int last, int gw, int lane) {
  const int G = pv.G, g = lane >> 2, t = lane & 3;
  float l0 = S.l[0], l1 = S.l[1], z0 = S.z[0], z1 = S.z[1];
#pragma unroll
  for (int s = 4; s <= 16; s <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, s);
    l1 += __shfl_xor_sync(0xffffffffu, l1, s);
    z0 += __shfl_xor_sync(0xffffffffu, z0, s);
    z1 += __shfl_xor_sync(0xffffffffu, z1, s);
  }
  const int stride = part_stride(G);
  float* dst = a.part + ((size_t)u * a.max_parts + (gw - first)) * stride;
#pragma unroll
  for (int mt = 0; mt < 8; mt++) {
    const int f = 16 * g + 2 * mt;
    if (2 * t < G) *reinterpret_cast<float2*>(dst + (2 * t) * kD + f) = make_float2(S.o[mt][0] + z0, S.o[mt][2] + z0);
    if (2 * t + 1 < G)
      *reinterpret_cast<float2*>(dst + (2 * t + 1) * kD + f) = make_float2(S.o[mt][1] + z1, S.o[mt][3] + z1);
  }
  if (g == 0) {
    if (2 * t < G) { dst[G * kD + 2 * t] = S.m[0]; dst[G * kD + kMaxG + 2 * t] = l0; }
    if (2 * t + 1 < G) { dst[G * kD + 2 * t + 1] = S.m[1]; dst[G * kD + kMaxG + 2 * t + 1] = l1; }
  }
  __threadfence();
  __syncwarp();
  int prev = 0;
  if (lane == 0) prev = atomicAdd(&a.done[u], 1);
  prev = __shfl_sync(0xffffffffu, prev, 0);
  const int nparts = last - first + 1;
  if (prev != nparts - 1) return;
  __threadfence();
  const float* src = a.part + (size_t)u * a.max_parts * stride;
  const int i = u / pv.hkv, kvh = u % pv.hkv;
  for (int qh = 0; qh < G; qh++) {
    float M = -INFINITY;
    for (int sp = 0; sp < nparts; sp++) M = fmaxf(M, __ldcg(src + sp * stride + G * kD + qh));
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    float Lsum = 0.0f;
    if (M != -INFINITY) {
      for (int sp = 0; sp < nparts; sp++) {
        const float ms = __ldcg(src + sp * stride + G * kD + qh);
        if (ms == -INFINITY) continue;
        const float w = exp2f(ms - M);
        const float4 o4 = __ldcg(reinterpret_cast<const float4*>(src + sp * stride + qh * kD) + lane);
        O.x += w * o4.x; O.y += w * o4.y; O.z += w * o4.z; O.w += w * o4.w;
        Lsum += w * __ldcg(src + sp * stride + G * kD + kMaxG + qh);
      }
    }
    const float inv = Lsum > 0.0f ? 1.0f / Lsum : 0.0f;
    reinterpret_cast<float4*>(a.out + ((size_t)i * pv.hkv * G + (size_t)kvh * G + qh) * kD)[lane] =
        make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
    if (lane == 0) a.lse2[(size_t)u * G + qh] = Lsum > 0.0f ? M + log2f(Lsum) : -INFINITY;
  }
  if (lane == 0) {
    a.done[u] = 0;
    if (a.update && kvh == 0) pv.rq(a.layer, sa.slots[i])[3] += 1;
  }
}

// Prefix over the call's heads of their work items (pages or chunks), in
// shared memory; every CTA computes the same. Returns the total.
__device__ int item_prefix(const PoolView& pv, const SlotArgs& sa, int layer, bool paged, int* s_pref, int* s_warp) {
  const int n_units = sa.n * pv.hkv;
  const int per = (n_units + blockDim.x - 1) / blockDim.x;
  const int u0 = min(n_units, (int)threadIdx.x * per), u1 = min(n_units, u0 + per);
  int sum = 0;
  for (int u = u0; u < u1; u++) {
    const int* cn = pv.cnt(layer, sa.slots[u / pv.hkv], u % pv.hkv);
    // paged: pages weighted by their chunks (T / 16); chunked: chunks
    const int items = paged ? (cn[0] + pv.hi.t - 1) / pv.hi.t * (pv.hi.t / kChunk) +
                                  (cn[1] + pv.lo.t - 1) / pv.lo.t * (pv.lo.t / kChunk)
                            : (cn[0] + kChunk - 1) / kChunk + (cn[1] + kChunk - 1) / kChunk;
    s_pref[u] = items;
    sum += items;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = sum;
#pragma unroll
  for (int s = 1; s < 32; s <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, s);
    if (lane >= s) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  int run = x - sum;
  for (int w = 0; w < warp; w++) run += s_warp[w];
  for (int u = u0; u < u1; u++) {
    const int v = s_pref[u];
    s_pref[u] = run;
    run += v;
  }
  if (threadIdx.x == blockDim.x - 1) s_pref[n_units] = run;
  __syncthreads();
  return s_pref[n_units];
}

// Heads without any stored token get a zero output (CTA 0).
__device__ void zero_empty_heads(const PoolView& pv, const AttnArgs& a, const SlotArgs& sa, const int* s_pref) {
  const int n_units = sa.n * pv.hkv, G = pv.G;
  for (int u = 0; u < n_units; u++) {
    if (s_pref[u + 1] != s_pref[u]) continue;
    const int i = u / pv.hkv, kvh = u % pv.hkv;
    for (int x = threadIdx.x; x < G * kD; x += blockDim.x)
      a.out[((size_t)i * pv.hkv * G + (size_t)kvh * G) * kD + x] = 0.0f;
    if (threadIdx.x < G) a.lse2[(size_t)u * G + threadIdx.x] = -INFINITY;
    if (threadIdx.x == 0 && a.update && kvh == 0) pv.rq(a.layer, sa.slots[i])[3] += 1;
  }
}

__device__ __forceinline__ int find_unit(const int* s_pref, int n_units, int g0) {
  int lo_u = 0, hi_u = n_units - 1;   // last u with s_pref[u] <= g0 (never an empty head)
  while (lo_u < hi_u) {
    const int mid = (lo_u + hi_u + 1) >> 1;
    if (s_pref[mid] <= g0) lo_u = mid; else hi_u = mid - 1;
  }
  return lo_u;
}

// ---------------------------------------------------------------------------
// Paged path: pages of T = 16k tokens (k = 1, 2), one bulk copy per page of
// its first four segments (K rows, V rows, K meta, V meta are contiguous at
// the page start). The work sequence is measured in chunks (a page weighs
// T/16); a warp takes the pages that start inside its range of chunks.
// ---------------------------------------------------------------------------
struct PageCursor {
  int u, begin, end;   // head and its chunk range
  int hp, np;          // hi pages, all pages
  int nh, nl;
  const int* row;
  int p, off;          // current page and its chunk offset
};

struct PagedCtx {
  const PoolView& pv;
  const SlotArgs& sa;
  const int* s_pref;
  int layer, n_units, wh, wl;

  __device__ __forceinline__ void at_unit(PageCursor& c, int u) const {
    c.u = u;
    c.begin = s_pref[u];
    c.end = s_pref[u + 1];
    const int* cn = pv.cnt(layer, sa.slots[u / pv.hkv], u % pv.hkv);
    c.nh = cn[0];
    c.nl = cn[1];
    c.hp = (c.nh + pv.hi.t - 1) / pv.hi.t;
    c.np = c.hp + (c.nl + pv.lo.t - 1) / pv.lo.t;
    c.row = pv.row(layer, sa.slots[u / pv.hkv], u % pv.hkv);
    c.p = 0;
    c.off = c.begin;
  }
  // move past pages of finished heads (and empty heads) while another head follows
  __device__ __forceinline__ void settle(PageCursor& c) const {
    while (c.p >= c.np && c.u + 1 < n_units) at_unit(c, c.u + 1);
  }
  __device__ __forceinline__ void next(PageCursor& c) const {
    c.off += c.p < c.hp ? wh : wl;
    c.p++;
    settle(c);
  }
  // first page starting at chunk offset >= x
  __device__ __forceinline__ void seek(PageCursor& c, int x) const {
    at_unit(c, find_unit(s_pref, n_units, x));
    const int o = x - c.begin;
    if (o > 0) {
      if (o <= c.hp * wh) {
        c.p = (o + wh - 1) / wh;
        c.off = c.begin + c.p * wh;
      } else {
        c.p = c.hp + (o - c.hp * wh + wl - 1) / wl;
        c.off = c.begin + c.hp * wh + (c.p - c.hp) * wl;
      }
    }
    settle(c);
  }
  __device__ __forceinline__ bool valid(const PageCursor& c, int g1) const { return c.p < c.np && c.off < g1; }
  // warps that own pages of head c.u (range width C)
  __device__ __forceinline__ void owners(const PageCursor& c, int C, int& first, int& last) const {
    first = c.begin / C;
    last = (c.end - (c.np > c.hp ? wl : wh)) / C;
  }
};

__global__ void __launch_bounds__(128, kCtasPerSm) k_attn_paged(PoolView pv, AttnArgs a, SlotArgs sa) {
  if (pv.noop()) return;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_warp[kAttnWarps];
  const int n_units = sa.n * pv.hkv;
  const int G = pv.G;
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem + kAttnWarps * kPageStages * a.stage_bytes);
  int* s_pref = reinterpret_cast<int*>(s_bar + kAttnWarps * kPageStages);
  const int total = item_prefix(pv, sa, a.layer, true, s_pref, s_warp);
  const int nwarps = gridDim.x * kAttnWarps;
  const int C = max(kMinChunks, (total + nwarps - 1) / nwarps);
  if (blockIdx.x == 0) zero_empty_heads(pv, a, sa, s_pref);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int gw = blockIdx.x * kAttnWarps + warp;
  const int g0 = gw * C, g1 = min(total, g0 + C);
  if (g0 >= g1) return;           // no block-wide barrier follows
  const PagedCtx ctx{pv, sa, s_pref, a.layer, n_units, pv.hi.t / kChunk, pv.lo.t / kChunk};
  PageCursor ci, cc;
  ctx.seek(ci, g0);
  if (!ctx.valid(ci, g1)) return;  // no page starts inside this range
  cc = ci;
  uint32_t bq_hi[8][2], bq_lo[8][2];
  float sq0, sq1;
  load_q(pv, a, cc.u / pv.hkv, cc.u % pv.hkv, g, t, bq_hi, bq_lo, sq0, sq1);
  uint8_t* wst = smem + warp * (kPageStages * a.stage_bytes);
  const uint32_t bar0 = smem_u32(s_bar + warp * kPageStages);
  if (lane == 0) {
    for (int st = 0; st < kPageStages; st++) mbar_init(bar0 + 8 * st, 1);
    fence_mbar_init();
    fence_proxy_async();
  }
  __syncwarp();
  int issued = 0;
  // one lane copies the next page's K | V | K meta | V meta prefix
  auto try_issue = [&]() {
    if (!ctx.valid(ci, g1)) return;
    if (lane == 0) {
      const int st = issued % kPageStages;
      const bool hi = ci.p < ci.hp;
      const TierGeom& tg = hi ? pv.hi : pv.lo;
      const int e = hi ? ci.p : pv.L - 1 - (ci.p - ci.hp);
      const uint32_t bar = bar0 + 8 * st;
      const uint32_t bytes = tg.off[4];
      mbar_expect_tx(bar, bytes);
      bulk_g2s(smem_u32(wst + st * a.stage_bytes), pv.page(__ldg(ci.row + e)), bytes, bar);
    }
    issued++;
    ctx.next(ci);
  };
  AttnState S;
  S.reset();
  for (int x = 0; x < kPageStages - 1; x++) try_issue();
  int cur_u = cc.u;
  for (int x = 0; x < issued; x++) {
    __syncwarp();                 // every lane is done with the stage being refilled
    fence_proxy_async();
    try_issue();
    if (!mbar_wait_bounded(bar0 + 8 * (x % kPageStages), (x / kPageStages) & 1)) {
      if (lane == 0 && atomicCAS(&pv.ctl->error, 0, DKV_ERR_TIMEOUT) == 0) pv.ctl->error_info = cc.u;
      for (int y = x + 1; y < min(issued, x + kPageStages); y++)
        mbar_wait_bounded(bar0 + 8 * (y % kPageStages), (y / kPageStages) & 1);
      return;
    }
    if (cc.u != cur_u) {          // the range crosses into the next head
      PageCursor prev = cc;
      ctx.at_unit(prev, cur_u);
      int first, last;
      ctx.owners(prev, C, first, last);
      publish(pv, a, sa, S, cur_u, first, last, gw, lane);
      cur_u = cc.u;
      load_q(pv, a, cc.u / pv.hkv, cc.u % pv.hkv, g, t, bq_hi, bq_lo, sq0, sq1);
      S.reset();
    }
    const bool hi = cc.p < cc.hp;
    const TierGeom& tg = hi ? pv.hi : pv.lo;
    const int pt = hi ? cc.p : cc.p - cc.hp;             // page index within the tier
    const int count = (hi ? cc.nh : cc.nl) - pt * tg.t;  // valid slots from this page's start
    const uint8_t* sb = wst + (x % kPageStages) * a.stage_bytes;
    const int jA = chunk_slot(g), jB = chunk_slot(g + 8);
    const int n_chunks = tg.t / kChunk;
    const int chunk0 = hi ? pt * n_chunks : (cc.nh + kChunk - 1) / kChunk + pt * n_chunks;
    for (int c = 0; c < n_chunks && c * kChunk < count; c++) {
      const int sA = c * kChunk + jA, sB = c * kChunk + jB;
      const uint8_t* kA = sb + sA * tg.kbytes + (hi ? 32 * t : 16 * t);
      const uint8_t* kB = sb + sB * tg.kbytes + (hi ? 32 * t : 16 * t);
      const uint8_t* v0 = hi ? sb + tg.off[1] + (c * 8 + 2 * t) * 128 + 16 * g : sb + tg.off[1] + (c * 4 + t) * 128 + 16 * g;
      const uint8_t* v1 = v0 + 128;
      const uint32_t kmA = *reinterpret_cast<const uint32_t*>(sb + tg.off[2] + 4 * sA);
      const uint32_t kmB = *reinterpret_cast<const uint32_t*>(sb + tg.off[2] + 4 * sB);
      const uint32_t vmA = *reinterpret_cast<const uint32_t*>(sb + tg.off[3] + 4 * sA);
      const uint32_t vmB = *reinterpret_cast<const uint32_t*>(sb + tg.off[3] + 4 * sB);
      float* lg = a.update ? a.logit + ((size_t)cc.u * a.max_chunks + chunk0 + c) * (kChunk * 8) : nullptr;
      attend_chunk(S, hi, kA, kB, v0, v1, kmA, kmB, vmA, vmB, sA < count, sB < count, bq_hi, bq_lo, sq0, sq1, lg,
                   G, g, t);
    }
    ctx.next(cc);
  }
  {
    PageCursor prev = cc;
    ctx.at_unit(prev, cur_u);
    int first, last;
    ctx.owners(prev, C, first, last);
    publish(pv, a, sa, S, cur_u, first, last, gw, lane);
  }
}

// ---------------------------------------------------------------------------
// Chunked path, any page geometry: work item = one 16-slot chunk, staged as
// the chunk's runs of K rows and V rows plus the meta segments of every page
// it touches (the copies spread over the lanes).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128, kCtasPerSm) k_attn_decode(PoolView pv, AttnArgs a, SlotArgs sa) {
  if (pv.noop()) return;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_warp[kAttnWarps];
  const int n_units = sa.n * pv.hkv;
  const int G = pv.G;
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem + kAttnWarps * kStages * a.stage_bytes);
  int* s_pref = reinterpret_cast<int*>(s_bar + kAttnWarps * kStages);
  const int total = item_prefix(pv, sa, a.layer, false, s_pref, s_warp);
  const int nwarps = gridDim.x * kAttnWarps;
  const int C = max(kMinChunks, (total + nwarps - 1) / nwarps);
  if (blockIdx.x == 0) zero_empty_heads(pv, a, sa, s_pref);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int gw = blockIdx.x * kAttnWarps + warp;
  const int g0 = gw * C, g1 = min(total, g0 + C);
  if (g0 >= g1) return;           // no block-wide barrier follows
  Cursor ci, cc;
  cursor_at(ci, find_unit(s_pref, n_units, g0), s_pref, pv, sa, a.layer, false);
  cursor_seek(ci, g0, s_pref, pv, sa, a.layer, false);
  cc = ci;
  uint32_t bq_hi[8][2], bq_lo[8][2];
  float sq0, sq1;
  load_q(pv, a, cc.u / pv.hkv, cc.u % pv.hkv, g, t, bq_hi, bq_lo, sq0, sq1);
  uint8_t* wst = smem + warp * (kStages * a.stage_bytes);
  const uint32_t bar0 = smem_u32(s_bar + warp * kStages);
  if (lane == 0) {
    for (int st = 0; st < kStages; st++) mbar_init(bar0 + 8 * st, 1);
    fence_mbar_init();
    fence_proxy_async();
  }
  __syncwarp();
  auto issue = [&](int x) {
    cursor_seek(ci, x, s_pref, pv, sa, a.layer, false);
    const int st = (x - g0) % kStages;
    const uint32_t sb = smem_u32(wst + st * a.stage_bytes);
    const uint32_t bar = bar0 + 8 * st;
    const int lc = x - ci.begin;
    const bool hi = lc < ci.hi_items;
    const int base = (hi ? lc : lc - ci.hi_items) * kChunk;
    const int n = min(kChunk, (hi ? ci.nh : ci.nl) - base);
    const TierGeom& tg = hi ? pv.hi : pv.lo;
    const int d0 = tg.div(base), npg = tg.div(base + n - 1) - d0 + 1;
    const int gsz = hi ? 2 : 4;            // slots per value row
    const void* src[2] = {nullptr, nullptr};
    uint32_t dst[2] = {0, 0}, bytes[2] = {0, 0};
    uint32_t tot = 0;
#pragma unroll
    for (int k = 0; k < 2; k++) {
      const int c = lane + 32 * k;
      if (c < 4 * npg) {
        const int r = c >> 2, kind = c & 3, d = d0 + r;
        const uint8_t* page = pv.page(__ldg(ci.row + (hi ? d : pv.L - 1 - d)));
        const int start = max(base, d * tg.t), end = min(base + n, (d + 1) * tg.t);
        const int ia = start - d * tg.t, ib = end - d * tg.t;
        if (kind == 0) {
          src[k] = page + tg.off[0] + ia * tg.kbytes;
          dst[k] = sb + (start - base) * tg.kbytes;
          bytes[k] = (ib - ia) * tg.kbytes;
        } else if (kind == 1) {
          const int r0 = ia / gsz, r1 = (ib + gsz - 1) / gsz;
          src[k] = page + tg.off[1] + r0 * 128;
          dst[k] = sb + kOffV + ((start - base) / gsz) * 128;
          bytes[k] = (r1 - r0) * 128;
        } else {
          src[k] = page + tg.off[kind];
          dst[k] = sb + kOffMeta + (kind - 2) * a.maxp * a.mseg + r * a.mseg;
          bytes[k] = (4 * tg.t + 15) & ~15;
        }
        tot += bytes[k];
      }
    }
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, s);
    if (lane == 0) mbar_expect_tx(bar, tot);
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 2; k++)
      if (bytes[k]) bulk_g2s(dst[k], src[k], bytes[k], bar);
  };
  AttnState S;
  S.reset();
  const int n = g1 - g0;
  for (int x = 0; x < kStages - 1 && x < n; x++) issue(g0 + x);
  for (int x = 0; x < n; x++) {
    if (x + kStages - 1 < n) {
      __syncwarp();               // every lane is done with the stage being refilled
      fence_proxy_async();
      issue(g0 + x + kStages - 1);
    }
    if (!mbar_wait_bounded(bar0 + 8 * (x % kStages), (x / kStages) & 1)) {
      if (lane == 0 && atomicCAS(&pv.ctl->error, 0, DKV_ERR_TIMEOUT) == 0) pv.ctl->error_info = cc.u;
      for (int y = x + 1; y < min(n, x + kStages); y++) mbar_wait_bounded(bar0 + 8 * (y % kStages), (y / kStages) & 1);
      return;
    }
    const int gx = g0 + x;
    if (gx >= cc.end) {           // the range crosses into the next head
      publish(pv, a, sa, S, cc.u, cc.begin / C, (cc.end - 1) / C, gw, lane);
      cursor_seek(cc, gx, s_pref, pv, sa, a.layer, false);
      load_q(pv, a, cc.u / pv.hkv, cc.u % pv.hkv, g, t, bq_hi, bq_lo, sq0, sq1);
      S.reset();
    }
    const int lc = gx - cc.begin;
    const bool hi = lc < cc.hi_items;
    const int base = (hi ? lc : lc - cc.hi_items) * kChunk;
    const int count = hi ? cc.nh : cc.nl;
    const uint8_t* sb = wst + (x % kStages) * a.stage_bytes;
    const TierGeom& tgc = hi ? pv.hi : pv.lo;
    const int d0c = tgc.div(base);
    const int jA = chunk_slot(g), jB = chunk_slot(g + 8);
    const int dA = tgc.div(base + jA), dB = tgc.div(base + jB);
    const uint8_t* mbase = sb + kOffMeta;
    const int mA = (dA - d0c) * a.mseg + 4 * (base + jA - dA * tgc.t);
    const int mB = (dB - d0c) * a.mseg + 4 * (base + jB - dB * tgc.t);
    const uint32_t kmA = *reinterpret_cast<const uint32_t*>(mbase + mA);
    const uint32_t kmB = *reinterpret_cast<const uint32_t*>(mbase + mB);
    const uint32_t vmA = *reinterpret_cast<const uint32_t*>(mbase + a.maxp * a.mseg + mA);
    const uint32_t vmB = *reinterpret_cast<const uint32_t*>(mbase + a.maxp * a.mseg + mB);
    const uint8_t* kA = sb + jA * tgc.kbytes + (hi ? 32 * t : 16 * t);
    const uint8_t* kB = sb + jB * tgc.kbytes + (hi ? 32 * t : 16 * t);
    const uint8_t* v0 = hi ? sb + kOffV + (2 * t) * 128 + 16 * g : sb + kOffV + t * 128 + 16 * g;
    const uint8_t* v1 = v0 + 128;
    float* lg = a.update ? a.logit + ((size_t)cc.u * a.max_chunks + lc) * (kChunk * 8) : nullptr;
    attend_chunk(S, hi, kA, kB, v0, v1, kmA, kmB, vmA, vmB, base + jA < count, base + jB < count, bq_hi, bq_lo,
                 sq0, sq1, lg, G, g, t);
  }
  publish(pv, a, sa, S, cc.u, cc.begin / C, (cc.end - 1) / C, gw, lane);
}

// Score update: every stored token's score gains max over the group's heads
// of its softmax probability, 2^(l2 - lse2).
__global__ void __launch_bounds__(256) k_attn_scores(PoolView pv, AttnArgs a, SlotArgs sa) {
  if (pv.noop()) return;
  const int unit = blockIdx.y, i = unit / pv.hkv, kvh = unit % pv.hkv;
  const int slot = sa.slots[i];
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
  const float* l2 = a.lse2 + (size_t)unit * G;
  float pm = 0.0f;
  for (int qh = 0; qh < G; qh++) pm = fmaxf(pm, exp2f(lg[qh] - l2[qh]));
  const int* row = pv.row(a.layer, slot, kvh);
  const TierGeom& tg = hi ? pv.hi : pv.lo;
  const int d = tg.div(s);
  uint8_t* pg = pv.page(row[hi ? d : pv.L - 1 - d]);
  float* sp = reinterpret_cast<float*>(pg + tg.off[4] + 4 * (s - d * tg.t));
  *sp = *sp + pm;
}

constexpr int kMaxAttnSmem = 220 * 1024;

// Pages a 16-slot chunk can touch for t tokens per page (chunks start at
// multiples of 16 slots).
static int pages_per_chunk(int t) {
  int m = 1;
  for (int c = 0; c < t; c++) {
    const int i0 = (c * kChunk) % t;
    m = std::max(m, (i0 + kChunk - 1) / t + 1);
  }
  return m;
}

cudaError_t launch_attention(Pool& P, int layer, const SlotArgs& sa, int max_tokens, const __half* q,
                             float* out, int update_scores, cudaStream_t st) {
  AttnArgs a;
  a.q = q;
  a.out = out;
  a.part = P.sc.apart;
  a.logit = P.sc.alogit;
  a.lse2 = P.sc.alse;
  a.done = P.sc.adone;
  a.max_parts = P.sc.max_splits;
  a.max_chunks = P.sc.max_chunks;
  a.update = update_scores;
  a.layer = layer;
  const int n_units = sa.n * P.pv.hkv;
  const bool paged = P.pv.hi.t % kChunk == 0 && P.pv.lo.t % kChunk == 0;
  int smem;
  if (paged) {
    a.mseg = 0;
    a.maxp = 1;
    a.stage_bytes = std::max(P.pv.hi.off[4], P.pv.lo.off[4]);
    smem = kAttnWarps * kPageStages * (a.stage_bytes + 8) + 4 * (n_units + 1);
  } else {
    a.mseg = (4 * std::max(P.pv.hi.t, P.pv.lo.t) + 15) & ~15;
    a.maxp = std::max(pages_per_chunk(P.pv.hi.t), pages_per_chunk(P.pv.lo.t));
    a.stage_bytes = kOffMeta + 2 * a.maxp * a.mseg;
    smem = kAttnWarps * kStages * (a.stage_bytes + 8) + 4 * (n_units + 1);
  }
  if (smem > kMaxAttnSmem) return cudaErrorInvalidConfiguration;
  if (paged)
    k_attn_paged<<<P.sm_count * kCtasPerSm, 128, smem, st>>>(P.pv, a, sa);
  else
    k_attn_decode<<<P.sm_count * kCtasPerSm, 128, smem, st>>>(P.pv, a, sa);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (update_scores) {
    const int max_chunks_call = (max_tokens + kChunk - 1) / kChunk + 1;
    const dim3 g2((max_chunks_call + 15) / 16, (unsigned)n_units);
    k_attn_scores<<<g2, 256, 0, st>>>(P.pv, a, sa);
    e = cudaGetLastError();
  }
  return e;
}

// ---------------------------------------------------------------------------
// Allocation-free variant (dkv_decode_attention_static). The same kernels
// work in one fixed device array instead of the pool's scratch: the merge
// counters, the per-head lse2, the per-warp partials and, with score updates,
// the per-chunk logits. The array is part of this library's device image; the
// CUDA driver reserves it when the module is loaded, so no call here
// allocates. Every call shares it and it keeps the last call's contents.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_attn_static_scratch[DKV_ATTN_STATIC_SCRATCH_BYTES];

constexpr int kMaxStaticDevices = 64;
static std::mutex g_static_mu;
static void* g_static_base[kMaxStaticDevices];

namespace {
size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Regions of the array for one call, each 256-byte aligned: merge counters
// at 0, then lse2, partials, logits. Strides are sized for the call's
// longest request, not the pool's maximum.
struct StaticLayout {
  size_t lse2, part, logit, total;
  int max_parts, max_chunks;
};

StaticLayout static_layout(int n_units, int G, int max_tokens, int update_scores) {
  StaticLayout L;
  L.max_chunks = (max_tokens + kChunk - 1) / kChunk + 1;
  L.max_parts = L.max_chunks / kMinChunks + 2;   // warps over one head (ranges >= kMinChunks)
  size_t off = round256((size_t)n_units * sizeof(int));
  L.lse2 = off;
  off = round256(off + (size_t)n_units * G * sizeof(float));
  L.part = off;
  off = round256(off + (size_t)n_units * L.max_parts * part_stride(G) * sizeof(float));
  L.logit = off;
  if (update_scores) off += (size_t)n_units * L.max_chunks * kChunk * 8 * sizeof(float);
  L.total = off;
  return L;
}

// Address of the array on the current device, looked up once per device.
cudaError_t static_scratch(int device, uint8_t** base) {
  if (device < 0 || device >= kMaxStaticDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_base[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_base[device] = p;
  }
  *base = static_cast<uint8_t*>(g_static_base[device]);
  return cudaSuccess;
}
}  // namespace

size_t attention_static_bytes(const Pool& P, int n_units, int max_tokens, int update_scores) {
  return static_layout(n_units, P.pv.G, max_tokens, update_scores).total;
}

cudaError_t launch_attention_static(Pool& P, int layer, const SlotArgs& sa, int max_tokens, const __half* q,
                                    float* out, int update_scores, cudaStream_t st) {
  const int n_units = sa.n * P.pv.hkv;
  const StaticLayout L = static_layout(n_units, P.pv.G, max_tokens, update_scores);
  if (L.total > DKV_ATTN_STATIC_SCRATCH_BYTES) return cudaErrorInvalidValue;
  uint8_t* base = nullptr;
  cudaError_t e = static_scratch(P.device, &base);
  if (e != cudaSuccess) return e;
  AttnArgs a;
  a.q = q;
  a.out = out;
  a.done = reinterpret_cast<int*>(base);
  a.lse2 = reinterpret_cast<float*>(base + L.lse2);
  a.part = reinterpret_cast<float*>(base + L.part);
  a.logit = reinterpret_cast<float*>(base + L.logit);
  a.max_parts = L.max_parts;
  a.max_chunks = L.max_chunks;
  a.update = update_scores;
  a.layer = layer;
  // The merge counters must start at zero. A finished call leaves them zero,
  // but one cut short (a wait that timed out) leaves some set.
  e = cudaMemsetAsync(a.done, 0, (size_t)n_units * sizeof(int), st);
  if (e != cudaSuccess) return e;
  const bool paged = P.pv.hi.t % kChunk == 0 && P.pv.lo.t % kChunk == 0;
  int smem;
  if (paged) {
    a.mseg = 0;
    a.maxp = 1;
    a.stage_bytes = std::max(P.pv.hi.off[4], P.pv.lo.off[4]);
    smem = kAttnWarps * kPageStages * (a.stage_bytes + 8) + 4 * (n_units + 1);
  } else {
    a.mseg = (4 * std::max(P.pv.hi.t, P.pv.lo.t) + 15) & ~15;
    a.maxp = std::max(pages_per_chunk(P.pv.hi.t), pages_per_chunk(P.pv.lo.t));
    a.stage_bytes = kOffMeta + 2 * a.maxp * a.mseg;
    smem = kAttnWarps * kStages * (a.stage_bytes + 8) + 4 * (n_units + 1);
  }
  if (smem > kMaxAttnSmem) return cudaErrorInvalidConfiguration;
  if (paged)
    k_attn_paged<<<P.sm_count * kCtasPerSm, 128, smem, st>>>(P.pv, a, sa);
  else
    k_attn_decode<<<P.sm_count * kCtasPerSm, 128, smem, st>>>(P.pv, a, sa);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (update_scores) {
    const dim3 g2((L.max_chunks + 15) / 16, (unsigned)n_units);
    k_attn_scores<<<g2, 256, 0, st>>>(P.pv, a, sa);
    e = cudaGetLastError();
  }
  return e;
}

cudaError_t configure_attention() {
  cudaError_t e = cudaFuncSetAttribute(k_attn_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxAttnSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_attn_paged, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxAttnSmem);
}

}  // namespace dkv
