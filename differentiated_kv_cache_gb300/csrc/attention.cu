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
// 1024 exponent, then the 1024 removed by hsub2/hfma2). P' enters the product
// as an fp16 pair plus its fp16 residual (for G <= 4 in the spare query
// columns 4..7, else in a second product).
//
// Work distribution: the sequences of all KV heads of the call are
// concatenated (pages weighted by their measured cost) and cut into equal
// contiguous ranges, one per warp of a persistent grid (the sequence split of
// the page's kernel, balanced). A warp writes a partial (m, l, O) for every
// head its range touches; the epilogue kernel, a programmatic dependent of
// the attention kernel, merges each head's partials and updates its scores.
// Data is staged in shared memory by bulk asynchronous copies completing on
// per-stage mbarriers:
//   k_attn_paged   pages of 16k tokens (chunk-aligned): one copy per page of
//                  its contiguous K | V | K-meta | V-meta | score prefix;
//   k_attn_decode  any page geometry: per 16-slot chunk, one copy per page run.
#include <algorithm>
#include <vector>

#include "dkv_kernels.cuh"

namespace dkv {

constexpr int kStages = 3;                 // ring depth per warp (chunked path)
constexpr int kPageStages = 3;             // ring depth per warp (paged path)
constexpr int kMinChunks = 8;              // ring work items per warp at least
// Attention warps per SM: on the paged path one CTA of 16 warps (four CTAs
// of 4 warps when 16 page rings do not fit in shared memory), on the chunked
// path four CTAs of 4 warps. With several CTAs per SM the warps of the CTA
// placed first are issued ahead of the others, so that the same work takes
// the fourth CTA 15 % longer (per-warp timelines on GB300); one CTA per SM
// has no such order among its warps.
constexpr int kWarpsPerSm = 16;
// Paged path: a page's share of a warp's range, in cost units: a fixed part
// for staging and bookkeeping plus a part per 16-slot chunk (from per-warp
// timelines on GB300: a lo page of two chunks takes 1.6 times a hi page at
// G = 4 and at G = 8).
__host__ __device__ __forceinline__ int page_cost(int G, int chunks) {
  return G <= 4 ? 3 + 4 * chunks : 3 + 5 * chunks;
}
// A head's items start with a fixed cost for the warp that enters it mid-range
// (the previous head's partial, the new queries): about one hi page.
__host__ __device__ __forceinline__ int head_cost(int G) { return G <= 4 ? 9 : 8; }
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
  float* logit;       // [unit][max_chunks][lrow]: chunk rows of [query < G][16 slots] log2-domain
                      // logits
  float* lse2;        // [unit][G]
  int victims;        // 1: the score update leaves victim-key partials in the pool
  int max_parts, max_chunks;
  int lrow;           // floats per chunk row: G * 16
  int nwarps;         // warps of the attention grid
  int update;
  int layer;
  int paged;          // 1: pages hold whole 16-slot chunks (k_attn_paged), 0: any geometry (k_attn_decode)
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
  // query of mma column g: with G <= 4 columns 4..7 repeat queries 0..3 (their
  // P.V columns carry the fp16 residuals of P')
  const int qg = G <= 4 ? (g & 3) : g;
  float qf[32];
  if (qg < G) {
    const uint4* qp = reinterpret_cast<const uint4*>(a.q + ((size_t)i * pv.hkv * G + (size_t)kvh * G + qg) * kD + 32 * t);
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

// Query fragments in the feature order of one tier's key rows (hi: 8-bit,
// lo: 4-bit) and the pre-scaled sums of queries 2t, 2t+1.
template <int GT>   // the group size when fixed at compile time, else 0 (pv.G)
__device__ __forceinline__ void load_q1(const PoolView& pv, const AttnArgs& a, int i, int kvh, int g, int t, bool hi,
                                        uint32_t (&bq)[8][2], float& sq0, float& sq1) {
  const int G = GT > 0 ? GT : pv.G;
  // query of mma column g: with G <= 4 columns 4..7 repeat queries 0..3 (their
  // P.V columns carry the fp16 residuals of P')
  const int qg = G <= 4 ? (g & 3) : g;
  float qf[32];
  if (qg < G) {
    const uint4* qp = reinterpret_cast<const uint4*>(a.q + ((size_t)i * pv.hkv * G + (size_t)kvh * G + qg) * kD + 32 * t);
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
  if (hi) {
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {
      bq[kk][0] = pack_half2(qf[4 * kk], qf[4 * kk + 1]);
      bq[kk][1] = pack_half2(qf[4 * kk + 2], qf[4 * kk + 3]);
    }
  } else {
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {
      const int w = kk >> 1, na = (kk & 1) ? 2 : 0;
      bq[kk][0] = pack_half2(qf[8 * w + na], qf[8 * w + na + 4]);
      bq[kk][1] = pack_half2(qf[8 * w + na + 1], qf[8 * w + na + 5]);
    }
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  const float sc = 1.4426950408889634f * rsqrtf((float)kD);
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
  if (lg != nullptr) {             // logit row of the chunk: [query][slot]
    const int jA = chunk_slot(g), jB = chunk_slot(g + 8);
    if (2 * t < G) {
      lg[(2 * t) * kChunk + jA] = l2[0];
      lg[(2 * t) * kChunk + jB] = l2[2];
    }
    if (2 * t + 1 < G) {
      lg[(2 * t + 1) * kChunk + jA] = l2[1];
      lg[(2 * t + 1) * kChunk + jB] = l2[3];
    }
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
  // P' as fp16 pairs plus their fp16 residuals: with G <= 4 the residuals take
  // the spare query columns 4..7 (threads t >= 2), else a second P.V product
  uint32_t h0, l0, h1, l1;
  split_half2(p0 * svA, p1 * svA, h0, l0);
  split_half2(p2 * svB, p3 * svB, h1, l1);
  const bool two = G > 4, res = !two && t >= 2;
  const uint32_t pb0 = movmatrix_trans(res ? l0 : h0), pb1 = movmatrix_trans(res ? l1 : h1);
  const uint32_t pr0 = two ? movmatrix_trans(l0) : 0u, pr1 = two ? movmatrix_trans(l1) : 0u;
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
      if (two) mma16816(S.o[mt], af, pr0, pr1);
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
      if (two) mma16816(S.o[mt], af, pr0, pr1);
    }
  }
}

// Width C of each attention warp's range of the work sequence (cost units on
// the paged path, chunks on the chunked path). The warps whose ranges hold a
// page (a chunk) of head u are first = (s_pref[u] + hw) / C (its first page
// starts hw after its items) to last = (offset of its last page) / C; a
// warp's partial of head u is record (warp - first) of the head.
__host__ __device__ __forceinline__ int range_width(int total, int nwarps, bool paged, int wh, int wl) {
  const int per = (total + nwarps - 1) / nwarps;
  const int lo = paged ? kMinChunks * (wh > wl ? wh : wl) : kMinChunks;
  return per > lo ? per : lo;
}

// Publish the warp's partial of head u: O^T (with the value-zero sums added),
// the running maxima and sums of queries 0..G-1, at index gw - first of the
// head's partials (warp ranges first..last cover the head). The merge runs in
// the epilogue kernel once every warp is done.
template <int GT>   // the group size when fixed at compile time, else 0 (pv.G)
__device__ __forceinline__ void publish(const PoolView& pv, const AttnArgs& a, AttnState& S, int u, int first, int gw,
                                        int lane) {
  const int G = GT > 0 ? GT : pv.G, g = lane >> 2, t = lane & 3;
  if (G <= 4) {                   // the residual columns (threads t ^ 2) into the query columns
#pragma unroll
    for (int mt = 0; mt < 8; mt++)
#pragma unroll
      for (int x = 0; x < 4; x++) S.o[mt][x] += __shfl_xor_sync(0xffffffffu, S.o[mt][x], 2);
  }
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
}

// Work items of a head with nh hi, nl lo and nm mid tokens: on the paged
// path its pages weighted by their cost (wh, wl, wm) after the head's own
// (hw), on the chunked path (two-tier pools only) its chunks.
__device__ __forceinline__ int head_items(const PoolView& pv, int nh, int nl, int nm, bool paged, int wh, int wl,
                                          int wm, int hw) {
  return paged ? (nh + nl + nm > 0 ? hw : 0) + (nh + pv.hi.t - 1) / pv.hi.t * wh +
                     (nl + pv.lo.t - 1) / pv.lo.t * wl + (nm > 0 ? (nm + pv.mid.t - 1) / pv.mid.t * wm : 0)
               : (nh + kChunk - 1) / kChunk + (nl + kChunk - 1) / kChunk;
}

// mid tokens of a head (MID: a three-tier pool; 0 in a two-tier pool)
template <bool MID>
__device__ __forceinline__ int mid_count(const int* cn) { return MID ? cn[4] : 0; }

// Prefix over the call's heads of their work items (pages or chunks), in
// shared memory; every CTA computes the same. Returns the total.
template <bool MID>
__device__ int item_prefix(const PoolView& pv, const SlotArgs& sa, int layer, bool paged, int wh, int wl, int wm,
                           int hw, int* s_pref, int* s_warp) {
  const int n_units = sa.n * pv.hkv;
  const int per = (n_units + blockDim.x - 1) / blockDim.x;
  const int u0 = min(n_units, (int)threadIdx.x * per), u1 = min(n_units, u0 + per);
  int sum = 0;
  for (int u = u0; u < u1; u++) {
    const int* cn = pv.cnt(layer, sa.slots[u / pv.hkv], u % pv.hkv);
    const int items = head_items(pv, cn[0], cn[1], mid_count<MID>(cn), paged, wh, wl, wm, hw);
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

__device__ __forceinline__ int find_unit(const int* s_pref, int n_units, int g0) {
  int lo_u = 0, hi_u = n_units - 1;   // last u with s_pref[u] <= g0 (never an empty head)
  while (lo_u < hi_u) {
    const int mid = (lo_u + hi_u + 1) >> 1;
    if (s_pref[mid] <= g0) lo_u = mid; else hi_u = mid - 1;
  }
  return lo_u;
}

// ---------------------------------------------------------------------------
// Paged path: pages of T = 16k tokens (k = 1, 2, ...), one bulk copy per page
// of its first five segments (K rows, V rows, K meta, V meta, scores are
// contiguous at the page start). The work sequence is measured in cost units
// (a page weighs page_cost(G, T/16), a head starts with head_cost(G)); a warp
// takes the pages that start inside its range, walked in batches of 32 pages
// one per lane into a table of page descriptors. The softmax rescales lazily: a group's
// probabilities are taken against the running maximum as long as no logit
// exceeds it by more than kLazy (log2 units), so that the cross-lane maximum
// and the rescale of O run only when the maximum really moves.
// ---------------------------------------------------------------------------
constexpr float kNegBig = -1.0e30f;   // running maximum before the first token
constexpr float kLazy = 8.0f;         // probabilities stay below 2^kLazy

struct PageCursor {
  int u, begin, end;   // head and its cost range
  int hp, mp, np;      // hi pages, mid pages (three-tier pools), all pages
  int nh, nl;
  const int* row;
  int p, off;          // current page and its cost offset
};

// A head's pages in the order the warps stream them: hi, mid (three-tier
// pools, MID), then lo.
template <bool MID>
struct PagedCtx {
  const PoolView& pv;
  const SlotArgs& sa;
  const int* s_pref;
  int layer, n_units, wh, wl, wm, hw;

  __device__ __forceinline__ void at_unit(PageCursor& c, int u) const {
    c.u = u;
    c.begin = s_pref[u];
    c.end = s_pref[u + 1];
    const int* cn = pv.cnt(layer, sa.slots[u / pv.hkv], u % pv.hkv);
    c.nh = cn[0];
    c.nl = cn[1];
    const int nm = mid_count<MID>(cn);
    c.hp = (c.nh + pv.hi.t - 1) / pv.hi.t;
    c.mp = nm > 0 ? (nm + pv.mid.t - 1) / pv.mid.t : 0;
    c.np = c.hp + c.mp + (c.nl + pv.lo.t - 1) / pv.lo.t;
    c.row = pv.row(layer, sa.slots[u / pv.hkv], u % pv.hkv);
    c.p = 0;
    c.off = c.begin + hw;
  }
  // move past pages of finished heads (and empty heads) while another head follows
  __device__ __forceinline__ void settle(PageCursor& c) const {
    while (c.p >= c.np && c.u + 1 < n_units) at_unit(c, c.u + 1);
  }
  // first page starting at cost offset >= x
  __device__ __forceinline__ void seek(PageCursor& c, int x) const {
    at_unit(c, find_unit(s_pref, n_units, x));
    const int o = x - c.off;        // from the head's first page
    if (o > 0) {
      if (o <= c.hp * wh) {
        c.p = (o + wh - 1) / wh;
        c.off += c.p * wh;
      } else if (o <= c.hp * wh + c.mp * wm) {
        c.p = c.hp + (o - c.hp * wh + wm - 1) / wm;
        c.off += c.hp * wh + (c.p - c.hp) * wm;
      } else {
        c.p = c.hp + c.mp + (o - c.hp * wh - c.mp * wm + wl - 1) / wl;
        c.off += c.hp * wh + c.mp * wm + (c.p - c.hp - c.mp) * wl;
      }
    }
    settle(c);
  }
  __device__ __forceinline__ bool valid(const PageCursor& c, int g1) const { return c.p < c.np && c.off < g1; }
  // first warp that owns pages of head u (range width C)
  __device__ __forceinline__ int first_owner(int u, int C) const { return (s_pref[u] + hw) / C; }
};

__device__ __forceinline__ void lazy_reset(AttnState& S) {
#pragma unroll
  for (int mt = 0; mt < 8; mt++)
#pragma unroll
    for (int x = 0; x < 4; x++) S.o[mt][x] = 0.0f;
  S.m[0] = S.m[1] = kNegBig;
  S.l[0] = S.l[1] = 0.0f;
  S.z[0] = S.z[1] = 0.0f;
}

__device__ __forceinline__ float lo_half(uint32_t w) { return __half2float(__ushort_as_half((uint16_t)w)); }
__device__ __forceinline__ float hi_half(uint32_t w) { return __half2float(__ushort_as_half((uint16_t)(w >> 16))); }

// NC consecutive chunks c0 .. c0+NC-1 of a staged page, one softmax step.
// FULL: every slot of the chunks is valid (no masking). KB, VB: the tier's
// key and value bits (hi 8/4, mid 8/2, lo 4/2).
template <int KB, int VB, int NC, bool FULL>
__device__ __forceinline__ void attend_chunks(AttnState& S, const uint8_t* sb, const TierGeom& tg, int c0, int count,
                                              const uint32_t (&bq)[8][2], float sq0, float sq1, float* lg, int lrow,
                                              int pid, int G, int g, int t, int jA, int jB) {
  constexpr float sc = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
  float l2[NC][4];
  uint32_t vm[NC][2];
#pragma unroll
  for (int c = 0; c < NC; c++) {
    const int sA = (c0 + c) * kChunk + jA, sB = (c0 + c) * kChunk + jB;
    float acc0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, acc1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (KB == 8) {
      const uint4* pa = reinterpret_cast<const uint4*>(sb + sA * 128 + 32 * t);
      const uint4* pb = reinterpret_cast<const uint4*>(sb + sB * 128 + 32 * t);
      const uint4 ka0 = pa[0], ka1 = pa[1], kb0 = pb[0], kb1 = pb[1];
      const uint32_t kaw[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
      const uint32_t kbw[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
#pragma unroll
      for (int kk = 0; kk < 8; kk++) {
        uint32_t af[4];
        af[0] = cvt_k8(kaw[kk], 0x4140u);
        af[1] = cvt_k8(kbw[kk], 0x4140u);
        af[2] = cvt_k8(kaw[kk], 0x4342u);
        af[3] = cvt_k8(kbw[kk], 0x4342u);
        mma16816((kk & 1) ? acc1 : acc0, af, bq[kk][0], bq[kk][1]);
      }
    } else {
      const uint4 ka = *reinterpret_cast<const uint4*>(sb + sA * 64 + 16 * t);
      const uint4 kb = *reinterpret_cast<const uint4*>(sb + sB * 64 + 16 * t);
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
        mma16816((kk & 1) ? acc1 : acc0, af, bq[kk][0], bq[kk][1]);
      }
    }
    const uint32_t kmA = *reinterpret_cast<const uint32_t*>(sb + tg.off[2] + 4 * sA);
    const uint32_t kmB = *reinterpret_cast<const uint32_t*>(sb + tg.off[2] + 4 * sB);
    vm[c][0] = *reinterpret_cast<const uint32_t*>(sb + tg.off[3] + 4 * sA);
    vm[c][1] = *reinterpret_cast<const uint32_t*>(sb + tg.off[3] + 4 * sB);
    const float skA = lo_half(kmA) * sc, zkA = hi_half(kmA), skB = lo_half(kmB) * sc, zkB = hi_half(kmB);
    l2[c][0] = __fmaf_rn(acc0[0] + acc1[0], skA, zkA * sq0);
    l2[c][1] = __fmaf_rn(acc0[1] + acc1[1], skA, zkA * sq1);
    l2[c][2] = __fmaf_rn(acc0[2] + acc1[2], skB, zkB * sq0);
    l2[c][3] = __fmaf_rn(acc0[3] + acc1[3], skB, zkB * sq1);
    if (!FULL) {
      if (sA >= count) l2[c][0] = l2[c][1] = -INFINITY;
      if (sB >= count) l2[c][2] = l2[c][3] = -INFINITY;
    }
    if (lg != nullptr) {           // scratch row of the chunk: its logits
      float* lc = lg + c * lrow;
      if (2 * t < G) {
        lc[(2 * t) * kChunk + jA] = l2[c][0];
        lc[(2 * t) * kChunk + jB] = l2[c][2];
      }
      if (2 * t + 1 < G) {
        lc[(2 * t + 1) * kChunk + jA] = l2[c][1];
        lc[(2 * t + 1) * kChunk + jB] = l2[c][3];
      }
    }
  }
  // ---- lazy online softmax over the NC chunks ----
  float cm0 = fmaxf(l2[0][0], l2[0][2]), cm1 = fmaxf(l2[0][1], l2[0][3]);
#pragma unroll
  for (int c = 1; c < NC; c++) {
    cm0 = fmaxf(cm0, fmaxf(l2[c][0], l2[c][2]));
    cm1 = fmaxf(cm1, fmaxf(l2[c][1], l2[c][3]));
  }
  if (__any_sync(0xffffffffu, cm0 > S.m[0] + kLazy || cm1 > S.m[1] + kLazy)) {
#pragma unroll
    for (int s = 4; s <= 16; s <<= 1) {
      cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, s));
      cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, s));
    }
    const float mn0 = fmaxf(S.m[0], cm0), mn1 = fmaxf(S.m[1], cm1);
    const float f0 = fast_exp2(S.m[0] - mn0), f1 = fast_exp2(S.m[1] - mn1);
    S.m[0] = mn0;
    S.m[1] = mn1;
    S.l[0] *= f0; S.z[0] *= f0;
    S.l[1] *= f1; S.z[1] *= f1;
#pragma unroll
    for (int mt = 0; mt < 8; mt++) {
      S.o[mt][0] *= f0; S.o[mt][2] *= f0;
      S.o[mt][1] *= f1; S.o[mt][3] *= f1;
    }
  }
  // v^ = s (c - off) + (z + off s), off = 8 (4-bit values) or 2 (2-bit values)
  constexpr float voff = VB == 4 ? 8.0f : 2.0f;
#pragma unroll
  for (int c = 0; c < NC; c++) {
    const float p0 = fast_exp2(l2[c][0] - S.m[0]), p1 = fast_exp2(l2[c][1] - S.m[1]);
    const float p2 = fast_exp2(l2[c][2] - S.m[0]), p3 = fast_exp2(l2[c][3] - S.m[1]);
    float svA = lo_half(vm[c][0]), svB = lo_half(vm[c][1]);
    float zvA = __fmaf_rn(voff, svA, hi_half(vm[c][0])), zvB = __fmaf_rn(voff, svB, hi_half(vm[c][1]));
    if (!FULL) {                   // meta of an unused slot may hold any bits
      const int sA = (c0 + c) * kChunk + jA, sB = (c0 + c) * kChunk + jB;
      if (sA >= count) svA = zvA = 0.0f;
      if (sB >= count) svB = zvB = 0.0f;
    }
    S.l[0] += p0 + p2;
    S.l[1] += p1 + p3;
    S.z[0] = __fmaf_rn(p0, zvA, __fmaf_rn(p2, zvB, S.z[0]));
    S.z[1] = __fmaf_rn(p1, zvA, __fmaf_rn(p3, zvB, S.z[1]));
    // P'^T as B fragments: block of tokens 0-7 and block of tokens 8-15
    // P' as fp16 pairs plus their fp16 residuals: with G <= 4 the residuals
    // take the spare query columns 4..7 (threads t >= 2), else a second P.V
    // product
    uint32_t h0, l0, h1, l1;
    split_half2(p0 * svA, p1 * svA, h0, l0);
    split_half2(p2 * svB, p3 * svB, h1, l1);
    const bool two = G > 4, res = !two && t >= 2;
    const uint32_t pb0 = movmatrix_trans(res ? l0 : h0), pb1 = movmatrix_trans(res ? l1 : h1);
    const uint32_t pr0 = two ? movmatrix_trans(l0) : 0u, pr1 = two ? movmatrix_trans(l1) : 0u;
    // ---- O^T += V^T . P'^T ----
    if (VB == 4) {
      const uint8_t* v0 = sb + tg.off[1] + ((c0 + c) * 8 + 2 * t) * 128 + 16 * g;
      const uint4 vq0 = *reinterpret_cast<const uint4*>(v0);
      const uint4 vq1 = *reinterpret_cast<const uint4*>(v0 + 128);
      const uint32_t vw0[4] = {vq0.x, vq0.y, vq0.z, vq0.w};
      const uint32_t vw1[4] = {vq1.x, vq1.y, vq1.z, vq1.w};
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
        if (two) mma16816(S.o[mt], af, pr0, pr1);
      }
    } else {
      const uint4 vq = *reinterpret_cast<const uint4*>(sb + tg.off[1] + ((c0 + c) * 4 + t) * 128 + 16 * g);
      const uint32_t vw[4] = {vq.x, vq.y, vq.z, vq.w};
#pragma unroll
      for (int mt = 0; mt < 8; mt++) {
        const uint32_t w = (mt & 1) ? vw[mt >> 1] >> 8 : vw[mt >> 1];
        uint32_t af[4];
        af[0] = cvv2_0(w);    // feature 16g+2mt,   slots e0,e1
        af[1] = cvv2_2(w);    // feature 16g+2mt+1, slots e0,e1
        af[2] = cvv2_1(w);    // feature 16g+2mt,   slots e2,e3
        af[3] = cvv2_3(w);    // feature 16g+2mt+1, slots e2,e3
        mma16816(S.o[mt], af, pb0, pb1);
        if (two) mma16816(S.o[mt], af, pr0, pr1);
      }
    }
  }
}

// All chunks of one staged page: pairs of chunks share a softmax step.
template <int KB, int VB>
__device__ __forceinline__ void attend_page(AttnState& S, const uint8_t* sb, const TierGeom& tg, int nch, int count,
                                            const uint32_t (&bq)[8][2], float sq0, float sq1, float* lg, int lrow,
                                            int pid, int G, int g, int t, int jA, int jB) {
  if (count >= nch * kChunk) {
    int c = 0;
    for (; c + 2 <= nch; c += 2)
      attend_chunks<KB, VB, 2, true>(S, sb, tg, c, count, bq, sq0, sq1, lg ? lg + c * lrow : nullptr, lrow, pid, G,
                                     g, t, jA, jB);
    if (c < nch)
      attend_chunks<KB, VB, 1, true>(S, sb, tg, c, count, bq, sq0, sq1, lg ? lg + c * lrow : nullptr, lrow, pid, G,
                                     g, t, jA, jB);
  } else {
    for (int c = 0; c * kChunk < count; c++)
      attend_chunks<KB, VB, 1, false>(S, sb, tg, c, count, bq, sq0, sq1, lg ? lg + c * lrow : nullptr, lrow, pid, G,
                                      g, t, jA, jB);
  }
}

// With score updates, every request of the call counts one more update (the
// importance denominator of the generation phase). Done by the attention
// kernel's first block after its wait, so that the whole epilogue, which
// waits for the attention grid, reads the advanced count.
__device__ __forceinline__ void count_update(const PoolView& pv, const AttnArgs& a, const SlotArgs& sa) {
  if (a.update && blockIdx.x == 0)
    for (int i = threadIdx.x; i < sa.n; i += blockDim.x) pv.rq(a.layer, sa.slots[i])[3] += 1;
}

// Tier tag of a page descriptor's count word (bit 31 hi, bit 30 mid).
constexpr uint32_t kDescHi = 0x80000000u, kDescMid = 0x40000000u;

// W: warps per CTA, 16 (one CTA per SM) or 4 (four CTAs per SM); GT: the
// group size when fixed at compile time (4, 8), else 0 (pv.G); MID: a
// three-tier pool (hi, mid and lo pages; the two-tier instances compile the
// mid tier out)
template <int W, int GT, bool MID>
__global__ void __launch_bounds__(32 * W, kWarpsPerSm / W) k_attn_paged(PoolView pv, AttnArgs a, SlotArgs sa) {
  // a programmatic dependent of the kernel before it (counts, pages); the
  // epilogue grid, which reads the counts before its own wait, may launch
  // once every block is past the wait
  if (!dependent_begin<true>(pv)) return;
  count_update(pv, a, sa);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_warp[W];
  const int n_units = sa.n * pv.hkv;
  const int G = GT > 0 ? GT : pv.G;
  const int nch_hi = pv.hi.t / kChunk, nch_lo = pv.lo.t / kChunk, nch_mid = MID ? pv.mid.t / kChunk : 0;
  const int wh = page_cost(G, nch_hi), wl = page_cost(G, nch_lo), hw = head_cost(G);
  const int wm = MID ? page_cost(G, nch_mid) : 0;
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem + W * kPageStages * a.stage_bytes);
  int4* s_tab = reinterpret_cast<int4*>(s_bar + W * kPageStages);   // [warp][2][32] page descriptors
  int* s_pref = reinterpret_cast<int*>(s_tab + W * 2 * 32);
  const int total = item_prefix<MID>(pv, sa, a.layer, true, wh, wl, wm, hw, s_pref, s_warp);
  const int nwarps = gridDim.x * W;
  // at least kMinChunks pages of the heaviest kind per range: a head is then
  // covered by at most (its pages / kMinChunks) + 2 ranges
  const int C = range_width(total, nwarps, true, wh, max(wl, wm));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int gw = blockIdx.x * W + warp;
  const int g0 = gw * C, g1 = min(total, g0 + C);
  const PagedCtx<MID> ctx{pv, sa, s_pref, a.layer, n_units, wh, wl, wm, hw};
  PageCursor ci;
  bool active = g0 < g1;
  if (active) {
    ctx.seek(ci, g0);
    active = ctx.valid(ci, g1);     // a page starts inside this range
  }
  uint8_t* wst = smem + warp * (kPageStages * a.stage_bytes);
  int4* wtab = s_tab + warp * 64;
  const uint32_t bar0 = smem_u32(s_bar + warp * kPageStages);
  if (!active) return;
  if (lane == 0) {
    for (int st = 0; st < kPageStages; st++) mbar_init(bar0 + 8 * st, 1);
    fence_mbar_init();
    fence_proxy_async();
  }
  __syncwarp();
  // The warp's pages in batches of 32, one page a lane: lane k of batch b
  // walks from the batch's first page (head bu, page bp of the head) k pages
  // on, across heads, and writes table entry (b & 1, k) = {head, page ID,
  // valid slots from the page start (bit 31: hi tier, bit 30: mid tier), the
  // head's chunk index of the page's first chunk}, or head -1 past the range.
  // The 32 page-ID loads are in flight together. Entries of batch b are
  // replaced by batch b + 2 only, after every page of batch b was consumed.
  int bu = ci.u, bp = ci.p;
  auto fill_batch = [&](int b) -> int {
    int u = bu, p = bp + lane;
    int nh = 0, nl = 0, nm = 0, hp = 0, mp = 0, np = 0;
    bool ok = true;
    for (;;) {
      const int* cn = pv.cnt(a.layer, sa.slots[u / pv.hkv], u % pv.hkv);
      nh = cn[0];
      nl = cn[1];
      hp = pv.hi.div(nh + pv.hi.t - 1);
      if (MID) {
        nm = cn[4];
        mp = nm > 0 ? pv.mid.div(nm + pv.mid.t - 1) : 0;
      }
      np = hp + mp + pv.lo.div(nl + pv.lo.t - 1);
      if (p < np) break;
      p -= np;
      if (++u >= n_units) {
        ok = false;
        break;
      }
    }
    const bool hi = p < hp, mid = MID && !hi && p < hp + mp;
    const int pt = hi ? p : (mid ? p - hp : p - hp - mp);
    if (ok) ok = s_pref[u] + hw + (hi ? pt * wh : (mid ? hp * wh + pt * wm : hp * wh + mp * wm + pt * wl)) < g1;
    int4 dsc = make_int4(-1, 0, 0, 0);
    if (ok) {
      const int count = hi ? nh - pt * pv.hi.t : (mid ? nm - pt * pv.mid.t : nl - pt * pv.lo.t);
      const int ch_h = (nh + kChunk - 1) / kChunk;
      const int chunk0 = hi ? pt * nch_hi
                            : (mid ? ch_h + pt * nch_mid : ch_h + (nm + kChunk - 1) / kChunk + pt * nch_lo);
      const int pid = __ldg(pv.row(a.layer, sa.slots[u / pv.hkv], u % pv.hkv) +
                            (hi ? pt : (mid ? pv.L + pt : pv.L - 1 - pt)));
      dsc = make_int4(u, pid, (int)((hi ? kDescHi : (mid ? kDescMid : 0u)) | (uint32_t)count), chunk0);
    }
    wtab[(b & 1) * 32 + lane] = dsc;
    const unsigned vm = __ballot_sync(0xffffffffu, ok);
    bu = __shfl_sync(0xffffffffu, u, 31);
    bp = __shfl_sync(0xffffffffu, p, 31) + 1;
    __syncwarp();
    return vm == 0xffffffffu ? 32 : __popc(vm);
  };
  // lane 0 copies page xi's K | V | K meta | V meta | score prefix into stage
  // xi % kPageStages
  auto issue = [&](int xi) {
    if (lane == 0) {
      const int4 dsc = wtab[((xi >> 5) & 1) * 32 + (xi & 31)];
      const int st = xi % kPageStages;
      const uint32_t bar = bar0 + 8 * st;
      const uint32_t bytes =
          dsc.z < 0 ? pv.hi.off[4] : (MID && (dsc.z & kDescMid) ? pv.mid.off[4] : pv.lo.off[4]);
      mbar_expect_tx(bar, bytes);
      bulk_g2s(smem_u32(wst + st * a.stage_bytes), pv.page(dsc.y), bytes, bar);
    }
  };
  int n_pages = fill_batch(0);    // pages known so far; a full batch may have successors
  bool more = n_pages == 32;
  for (int x = 0; x < kPageStages - 1 && x < n_pages; x++) issue(x);
  AttnState S;
  lazy_reset(S);
  // the first head's queries load while its first pages are in flight; the
  // 8-bit key order serves hi and mid pages, the 4-bit one lo pages
  uint32_t bq[8][2];
  float sq0, sq1;
  bool q_hi = ci.p < ci.hp + ci.mp;
  int cur_u = ci.u;
  load_q1<GT>(pv, a, cur_u / pv.hkv, cur_u % pv.hkv, g, t, q_hi, bq, sq0, sq1);
  const int jA = chunk_slot(g), jB = chunk_slot(g + 8);
  bool failed = false;
  for (int x = 0; x < n_pages; x++) {
    __syncwarp();                 // every lane is done with the stage being refilled
    fence_proxy_async();
    const int xi = x + kPageStages - 1;
    if (more && xi == n_pages) {  // the next batch
      const int v = fill_batch(xi >> 5);
      n_pages += v;
      more = v == 32;
    }
    if (xi < n_pages) issue(xi);
    if (!mbar_wait_bounded(bar0 + 8 * (x % kPageStages), (x / kPageStages) & 1)) {
      if (lane == 0 && atomicCAS(&pv.ctl->error, 0, DKV_ERR_TIMEOUT) == 0) pv.ctl->error_info = cur_u;
      for (int y = x + 1; y < min(n_pages, x + kPageStages); y++)
        mbar_wait_bounded(bar0 + 8 * (y % kPageStages), (y / kPageStages) & 1);
      failed = true;
      break;
    }
    const int4 d = wtab[((x >> 5) & 1) * 32 + (x & 31)];   // head, page ID, valid slots | tier, first chunk
    const bool hi = d.z < 0;
    const bool mid = MID && (d.z & kDescMid) != 0;
    const bool k8 = hi || mid;    // 8-bit keys
    const int count = d.z & 0x3fffffff;
    if (d.x != cur_u) {           // the range enters the next head
      publish<GT>(pv, a, S, cur_u, ctx.first_owner(cur_u, C), gw, lane);
      cur_u = d.x;
      q_hi = k8;
      load_q1<GT>(pv, a, cur_u / pv.hkv, cur_u % pv.hkv, g, t, k8, bq, sq0, sq1);
      lazy_reset(S);
    } else if (k8 != q_hi) {      // from the head's 8-bit-key pages to its lo pages
      q_hi = k8;
      load_q1<GT>(pv, a, cur_u / pv.hkv, cur_u % pv.hkv, g, t, k8, bq, sq0, sq1);
    }
    const uint8_t* sb = wst + (x % kPageStages) * a.stage_bytes;
    float* lgp = a.update ? a.logit + ((size_t)cur_u * a.max_chunks + d.w) * a.lrow : nullptr;
    if (hi)
      attend_page<8, 4>(S, sb, pv.hi, nch_hi, count, bq, sq0, sq1, lgp, a.lrow, d.y, G, g, t, jA, jB);
    else if (MID && mid)
      attend_page<8, 2>(S, sb, pv.mid, nch_mid, count, bq, sq0, sq1, lgp, a.lrow, d.y, G, g, t, jA, jB);
    else
      attend_page<4, 2>(S, sb, pv.lo, nch_lo, count, bq, sq0, sq1, lgp, a.lrow, d.y, G, g, t, jA, jB);
  }
  if (!failed) publish<GT>(pv, a, S, cur_u, ctx.first_owner(cur_u, C), gw, lane);
}

// ---------------------------------------------------------------------------
// Chunked path, any page geometry: work item = one 16-slot chunk, staged as
// the chunk's runs of K rows and V rows plus the meta segments of every page
// it touches (the copies spread over the lanes).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(32 * kAttnWarps, kWarpsPerSm / kAttnWarps) k_attn_decode(PoolView pv, AttnArgs a,
                                                                                          SlotArgs sa) {
  // a programmatic dependent of the kernel before it (counts, pages); the
  // epilogue grid, which reads the counts before its own wait, may launch
  // once every block is past the wait
  if (!dependent_begin<true>(pv)) return;
  count_update(pv, a, sa);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_warp[kAttnWarps];
  const int n_units = sa.n * pv.hkv;
  const int G = pv.G;
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem + kAttnWarps * kStages * a.stage_bytes);
  int* s_pref = reinterpret_cast<int*>(s_bar + kAttnWarps * kStages);
  const int total = item_prefix<false>(pv, sa, a.layer, false, 1, 1, 0, 0, s_pref, s_warp);
  const int nwarps = gridDim.x * kAttnWarps;
  const int C = range_width(total, nwarps, false, 1, 1);
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
      publish<0>(pv, a, S, cc.u, cc.begin / C, gw, lane);
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
    float* lg = a.update ? a.logit + ((size_t)cc.u * a.max_chunks + lc) * a.lrow : nullptr;
    attend_chunk(S, hi, kA, kB, v0, v1, kmA, kmB, vmA, vmB, base + jA < count, base + jB < count, bq_hi, bq_lo,
                 sq0, sq1, lg, G, g, t);
  }
  publish<0>(pv, a, S, cc.u, cc.begin / C, gw, lane);
}

// ---------------------------------------------------------------------------
// Epilogue of a decode-attention call, launched as a programmatic dependent of
// the attention kernel: the merge of each head's partials into out and lse2
// and, with score updates, every stored token's new score
//   S_j += max over the group's queries of 2^(l2_j - lse2).
// Grid (block, head), at most one wave of blocks. With score updates block x
// of a head takes its chunk steps x, x + nb, ... (EC chunks each): warp 0
// stages a step's scratch rows with one bulk copy; the head's merge tasks
// (task t of a head spread over nb blocks goes to block t mod nb; task =
// query t / 4, features 32 (t % 4) ..) run on the block's warps and, when
// every query has a task in the block, hand it the head's lse2 (else warp 0
// derives it from the partials); then every thread writes new scores.
// Without score updates the head's blocks share its merge tasks on all
// warps. Everything a block needs before the attention kernel completes (its
// head's counts and partial count in the attention kernels' range partition)
// it derives from the head counts while it waits.
// ---------------------------------------------------------------------------
constexpr int kEpiThreads = 256;
constexpr int kEpiWarps = kEpiThreads / 32;
static_assert(kEpiWarps == kVictimWarps, "one victim-key partial per epilogue warp");
constexpr int kSlices = kD / 32;             // merge tasks per query: feature slices of 32
constexpr int kMergeRegs = 4;                // partials per lane held in registers by a merge task

// chunks per epilogue step: 8 slots a thread for G <= 4, 4 above
__host__ __device__ constexpr int epi_chunks(int G) { return G <= 4 ? 128 : 64; }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, s));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) x += __shfl_xor_sync(0xffffffffu, x, s);
  return x;
}

// Shared-memory layout of the epilogue (bytes), the same on host and device:
// the step's chunk rows (score updates only), lse2 of the head, mbarrier.
struct EpiSmem {
  int rows, lse, misc, total;
  __host__ __device__ EpiSmem(int G, bool update) {
    rows = 0;
    lse = update ? epi_chunks(G) * G * kChunk * 4 : 0;
    misc = lse + 4 * kMaxG;
    total = misc + 16;
  }
};

// Items of head u in the attention kernels' partition (pages weighted by
// cost on the paged path, chunks on the chunked path): the offset of its
// first item and the total over the call, from one block-wide reduction over
// the heads' counts.
template <bool MID>
__device__ void head_span(const PoolView& pv, const SlotArgs& sa, int layer, bool paged, int wh, int wl, int wm,
                          int hw, int u, int* s_red, int& begin, int& total) {
  const int n_units = sa.n * pv.hkv;
  int before = 0, all = 0;
  for (int v = threadIdx.x; v < n_units; v += blockDim.x) {
    const int* cn = pv.cnt(layer, sa.slots[v / pv.hkv], v % pv.hkv);
    const int nh = __ldcg(cn), nl = __ldcg(cn + 1), nm = MID ? __ldcg(cn + 4) : 0;
    const int items = head_items(pv, nh, nl, nm, paged, wh, wl, wm, hw);
    all += items;
    if (v < u) before += items;
  }
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, s);
    all += __shfl_xor_sync(0xffffffffu, all, s);
  }
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    s_red[2 * warp] = before;
    s_red[2 * warp + 1] = all;
  }
  __syncthreads();
  begin = 0;
  total = 0;
  for (int w = 0; w < nw; w++) {
    begin += s_red[2 * w];
    total += s_red[2 * w + 1];
  }
}

// Merge task of head u (np partials): query qh, features 32 sl .. 32 sl + 31.
// Lane (quad q, group pg) sums partials pg, pg + 4, ... of feature quad q;
// every lane also takes partial `lane` (lane + 32, ...) for the query's
// maximum M and rescaled sum L. The loads of the first 16 partials (and of
// the first 32 for M and L) are all issued before any is used. lse_dst, when
// given, receives the query's lse2 (M + log2 L).
template <int G>
__device__ void merge_task(const PoolView& pv, const AttnArgs& a, const SlotArgs& sa, int u, int np, int qh, int sl,
                           int lane, float* lse_dst) {
  const int stride = part_stride(G);
  const float* src = a.part + (size_t)u * a.max_parts * stride;
  const int q = sl * 8 + (lane & 7), pg = lane >> 3;
  float4 o4[kMergeRegs];
  float mo[kMergeRegs];
#pragma unroll
  for (int r = 0; r < kMergeRegs; r++) {
    const int p = pg + 4 * r;
    o4[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    mo[r] = -INFINITY;
    if (p < np) {
      o4[r] = __ldcg(reinterpret_cast<const float4*>(src + (size_t)p * stride + qh * kD) + q);
      mo[r] = __ldcg(src + (size_t)p * stride + G * kD + qh);
    }
  }
  float ml = -INFINITY, ll = 0.0f;
  if (lane < np) {
    ml = __ldcg(src + (size_t)lane * stride + G * kD + qh);
    ll = __ldcg(src + (size_t)lane * stride + G * kD + kMaxG + qh);
  }
  float M = ml;
  for (int p = lane + 32; p < np; p += 32) M = fmaxf(M, __ldcg(src + (size_t)p * stride + G * kD + qh));
  M = warp_max(M);
  float L = ml != -INFINITY ? ll * fast_exp2(ml - M) : 0.0f;
  for (int p = lane + 32; p < np; p += 32) {
    const float ms = __ldcg(src + (size_t)p * stride + G * kD + qh);
    if (ms != -INFINITY) L += __ldcg(src + (size_t)p * stride + G * kD + kMaxG + qh) * fast_exp2(ms - M);
  }
  L = warp_sum(L);
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < kMergeRegs; r++) {
    const float w = mo[r] == -INFINITY ? 0.0f : fast_exp2(mo[r] - M);
    o.x += w * o4[r].x; o.y += w * o4[r].y; o.z += w * o4[r].z; o.w += w * o4[r].w;
  }
#pragma unroll 4
  for (int p = pg + 4 * kMergeRegs; p < np; p += 4) {   // heads of more than 16 partials
    const float ms = __ldcg(src + (size_t)p * stride + G * kD + qh);
    const float4 v = __ldcg(reinterpret_cast<const float4*>(src + (size_t)p * stride + qh * kD) + q);
    const float w = ms == -INFINITY ? 0.0f : fast_exp2(ms - M);
    o.x += w * v.x; o.y += w * v.y; o.z += w * v.z; o.w += w * v.w;
  }
#pragma unroll
  for (int s = 8; s <= 16; s <<= 1) {
    o.x += __shfl_xor_sync(0xffffffffu, o.x, s);
    o.y += __shfl_xor_sync(0xffffffffu, o.y, s);
    o.z += __shfl_xor_sync(0xffffffffu, o.z, s);
    o.w += __shfl_xor_sync(0xffffffffu, o.w, s);
  }
  const int i = u / pv.hkv, kvh = u % pv.hkv;
  if (pg == 0) {
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    reinterpret_cast<float4*>(a.out + ((size_t)i * pv.hkv * G + (size_t)kvh * G + qh) * kD)[q] =
        make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
  }
  if (lane == 0 && (sl == 0 || lse_dst != nullptr)) {
    const float lse2 = L > 0.0f ? M + log2f(L) : -INFINITY;
    if (lse_dst != nullptr) *lse_dst = lse2;
    if (sl == 0) a.lse2[(size_t)u * G + qh] = lse2;
  }
}

// lse2 of head u's G queries from its np partials (lane = partial; lanes fold
// partials beyond the 32nd in online), written to dst[0 .. G).
template <int G>
__device__ void head_lse(const AttnArgs& a, int u, int np, int lane, float* dst) {
  const int stride = part_stride(G);
  const float* src = a.part + (size_t)u * a.max_parts * stride + G * kD;
  float m[G], l[G];
#pragma unroll
  for (int qh = 0; qh < G; qh++) {
    m[qh] = -INFINITY;
    l[qh] = 0.0f;
  }
  if (lane < np) {
#pragma unroll
    for (int qh = 0; qh < G; qh++) {
      m[qh] = __ldcg(src + (size_t)lane * stride + qh);
      l[qh] = __ldcg(src + (size_t)lane * stride + kMaxG + qh);
    }
  }
  for (int p = lane + 32; p < np; p += 32) {
#pragma unroll
    for (int qh = 0; qh < G; qh++) {
      const float mp = __ldcg(src + (size_t)p * stride + qh), lp = __ldcg(src + (size_t)p * stride + kMaxG + qh);
      const float mn = fmaxf(m[qh], mp);
      l[qh] = l[qh] * fast_exp2(m[qh] - mn) + lp * fast_exp2(mp - mn);
      m[qh] = mn;
    }
  }
#pragma unroll
  for (int qh = 0; qh < G; qh++) {
    const float M = warp_max(m[qh]);
    const float L = warp_sum(m[qh] != -INFINITY ? l[qh] * fast_exp2(m[qh] - M) : 0.0f);
    if (lane == 0) dst[qh] = L > 0.0f ? M + log2f(L) : -INFINITY;
  }
}

// A head that stores no token: zero output (G rows) and lse2 = -inf, after
// the attention kernel, whose writes come first.
__device__ __noinline__ void empty_head(float* out, float* lse2, int G) {
  pdl_wait();
  for (int x = threadIdx.x; x < G * kD; x += blockDim.x) out[x] = 0.0f;
  if (threadIdx.x < G) lse2[threadIdx.x] = -INFINITY;
}


// Registers of a thread's slot positions per chunk step: four slots a
// chunk-quarter (paged) or one slot (chunked) per iteration; at most 8.
constexpr int kPosRegs = 8;
static_assert(epi_chunks(1) * kChunk / kEpiThreads <= kPosRegs, "position registers");

// Geometry and table entry of a tier's page (MID: the pool has the mid tier;
// a two-tier instance chooses between hi and lo only).
template <bool MID>
__device__ __forceinline__ const TierGeom& tier_geom(const PoolView& pv, int tier) {
  return MID ? pv.geom(tier) : (tier == kTierHi ? pv.hi : pv.lo);
}
template <bool MID>
__device__ __forceinline__ int tier_entry(const PoolView& pv, int tier, int k) {
  return MID ? pv.entry(tier, k) : (tier == kTierHi ? k : pv.L - 1 - k);
}

// The chunks of a head's epilogue rows: its hi chunks, then its mid chunks
// (three-tier pools, MID), then its lo chunks.
template <bool MID>
struct HeadChunks {
  int ch_hi, ch_mid, nh, nm, nl;
  // tier of chunk lc, the tier slot of its first row and the tier's tokens
  __device__ __forceinline__ int tier(int lc, int& slot0, int& n) const {
    if (lc < ch_hi) {
      slot0 = lc * kChunk;
      n = nh;
      return kTierHi;
    }
    if (MID && lc < ch_hi + ch_mid) {
      slot0 = (lc - ch_hi) * kChunk;
      n = nm;
      return kTierMid;
    }
    slot0 = (lc - ch_hi - ch_mid) * kChunk;
    n = nl;
    return kTierLo;
  }
};

// Positions of this thread's slots in chunk step `step` of the head, in the
// order the score-update loops visit them (0 where a slot is not stored),
// and on the paged path their scores before the update and each quad's page
// ID (vs, vd). Read from the pages through the table before the grid-
// dependency wait: the attention kernel changes neither (the scores are
// written by this epilogue only), and a page's score and position segments
// of a chunk share one 128-byte line.
template <int EC, bool MID>
__device__ __forceinline__ void load_positions(const PoolView& pv, const int* row_tab, bool paged, int step, int nch,
                                               const HeadChunks<MID>& hc, int* vp, float* vs, int* vd) {
  const int c0 = step * EC, c1 = min(nch, c0 + EC);
#pragma unroll
  for (int e = 0; e < kPosRegs; e++) vp[e] = 0;
  if (paged) {
#pragma unroll
    for (int k = 0; k < EC * kChunk / 4 / kEpiThreads; k++) {
      const int x = k * kEpiThreads + threadIdx.x;
      const int lc = c0 + (x >> 2), j0 = 4 * (x & 3);
      if (lc >= c1) break;
      int s0, n;
      const int tier = hc.tier(lc, s0, n);
      s0 += j0;
      if (s0 >= n) continue;
      const TierGeom& tg = tier_geom<MID>(pv, tier);
      const int d = tg.div(s0);
      const int pid = __ldg(row_tab + tier_entry<MID>(pv, tier, d));
      const int4 p = __ldcg(reinterpret_cast<const int4*>(pv.page(pid) + tg.off[5]) + ((s0 - d * tg.t) >> 2));
      const float4 o = __ldcg(reinterpret_cast<const float4*>(pv.page(pid) + tg.off[4]) + ((s0 - d * tg.t) >> 2));
      vp[4 * k] = p.x;
      vp[4 * k + 1] = p.y;
      vp[4 * k + 2] = p.z;
      vp[4 * k + 3] = p.w;
      vs[4 * k] = o.x;
      vs[4 * k + 1] = o.y;
      vs[4 * k + 2] = o.z;
      vs[4 * k + 3] = o.w;
      vd[k] = pid;
    }
  } else {
#pragma unroll
    for (int k = 0; k < EC * kChunk / kEpiThreads; k++) {
      const int x = k * kEpiThreads + threadIdx.x;
      const int lc = c0 + x / kChunk, j = x % kChunk;
      if (lc >= c1) break;
      int slot, n;
      const int tier = hc.tier(lc, slot, n);
      slot += j;
      if (slot >= n) continue;
      const TierGeom& tg = tier_geom<MID>(pv, tier);
      const int d = tg.div(slot);
      const int pid = __ldg(row_tab + tier_entry<MID>(pv, tier, d));
      vp[k] = __ldcg(reinterpret_cast<const int*>(pv.page(pid) + tg.off[5]) + (slot - d * tg.t));
    }
  }
}

template <int G, bool MID>
__global__ void __launch_bounds__(kEpiThreads, 4) k_attn_epi(PoolView pv, AttnArgs a, SlotArgs sa) {
  if (pv.noop()) return;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_red[2 * kEpiWarps];
  constexpr int EC = epi_chunks(G);
  const int u = blockIdx.y, xb = blockIdx.x;
  const int i = u / pv.hkv, kvh = u % pv.hkv;
  const bool paged = a.paged != 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int* cn = pv.cnt(a.layer, sa.slots[i], kvh);
  const int nh = __ldcg(cn), nl = __ldcg(cn + 1), nm = MID ? __ldcg(cn + 4) : 0;
  if (nh + nl + nm == 0) {        // an empty head: zero output, lse2 = -inf
    if (xb == 0)
      empty_head(a.out + ((size_t)i * pv.hkv + kvh) * G * kD, a.lse2 + (size_t)u * G, G);
    return;
  }
  const int ch_hi = (nh + kChunk - 1) / kChunk, ch_mid = MID ? (nm + kChunk - 1) / kChunk : 0;
  const int nch = ch_hi + ch_mid + (nl + kChunk - 1) / kChunk;
  const HeadChunks<MID> hc{ch_hi, ch_mid, nh, nm, nl};
  // blocks of the head: with score updates one per chunk step of EC chunks
  // up to the grid's width (block x takes steps x, x + nb, ...), else every
  // block
  const int nsteps = (nch + EC - 1) / EC;
  const int nb = a.update ? min(nsteps, (int)gridDim.x) : (int)gridDim.x;
  if (xb >= nb) return;
  // the head's partial count in the attention kernels' range partition
  const int wh = paged ? page_cost(G, pv.hi.t / kChunk) : 1;
  const int wl = paged ? page_cost(G, pv.lo.t / kChunk) : 1;
  const int wm = MID ? page_cost(G, pv.mid.t / kChunk) : 0;
  const int hw = paged ? head_cost(G) : 0;
  int begin, total;
  head_span<MID>(pv, sa, a.layer, paged, wh, wl, wm, hw, u, s_red, begin, total);
  const int items = head_items(pv, nh, nl, nm, paged, wh, wl, wm, hw);
  const int C = range_width(total, a.nwarps, paged, wh, max(wl, wm));
  const int first = (begin + hw) / C;
  // the partial of the warp that owns the head's last page (lo, else mid, else hi)
  const int last = paged ? (begin + items - (nl > 0 ? wl : (nm > 0 ? wm : wh))) / C : (begin + items - 1) / C;
  const int np = last - first + 1;
  const EpiSmem L(G, a.update != 0);
  // With score updates the block also leaves victim keys (pool scratch only);
  // the positions of its first step's slots load now, before the wait: the
  // table and the pages' position segments do not change in this call.
  const bool victims = a.update && a.victims && nb * kEpiWarps <= pv.max_vp;
  const int* row_tab = pv.row(a.layer, sa.slots[i], kvh);
  int vp[kPosRegs], vd[kPosRegs / 4];
  float vs[kPosRegs];
  if (a.update) load_positions<EC, MID>(pv, row_tab, paged, xb, nch, hc, vp, vs, vd);
  float* s_rows = reinterpret_cast<float*>(smem + L.rows);
  float* s_lse = reinterpret_cast<float*>(smem + L.lse);
  const uint32_t bar = smem_u32(smem + L.misc);
  if (a.update && threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  // partials and chunk rows: written by the attention kernel. A device error
  // it raised itself leaves this call's outputs undefined (the status says so)
  pdl_wait();
  // merge tasks of this block: tasks xb, xb + nb, ... of the head (task =
  // query x feature slice). With nb <= kSlices every query has a task in every
  // block, and the task of slice < nb hands the block its lse2; otherwise warp
  // 0 derives lse2 from the partials and the tasks run on warps 1..
  const bool own_lse = a.update && nb > kSlices;
  const int w0 = own_lse ? 1 : 0;
  if (a.update && warp == 0) {
    if (lane == 0) {              // the rows of the block's first step
      const int c0 = xb * EC, c1 = min(nch, c0 + EC);
      const uint32_t bytes = (uint32_t)(c1 - c0) * a.lrow * 4u;
      mbar_expect_tx(bar, bytes);
      bulk_g2s(smem_u32(s_rows), a.logit + ((size_t)u * a.max_chunks + c0) * a.lrow, bytes, bar);
    }
    if (own_lse) head_lse<G>(a, u, np, lane, s_lse);
  }
  if (warp >= w0) {
    int j = 0;
    for (int task = xb; task < G * kSlices; task += nb, j++)
      if (j % (kEpiWarps - w0) == warp - w0) {
        const int qh = task / kSlices, sl = task % kSlices;
        merge_task<G>(pv, a, sa, u, np, qh, sl, lane, a.update && !own_lse && sl < nb ? s_lse + qh : nullptr);
      }
  }
  if (!a.update) return;
  __syncthreads();                // s_lse
  // new scores of the block's slots: S_j += max over queries of 2^(l2 - lse2)
  float lse[G];
#pragma unroll
  for (int qh = 0; qh < G; qh++) lse[qh] = s_lse[qh];
  // Victim keys of the head's next generation step, from the new scores:
  // the step after this call has length N + 1, so t_c is position N - W and
  // hi victims lie before N + 1 - W. The update count was advanced by the
  // attention kernel, which this grid waited for.
  int vn0 = 0, vN = 0, vupd = 0;
  if (victims) {
    const int* rq = pv.rq(a.layer, sa.slots[i]);
    vn0 = __ldcg(rq + 1);
    vN = __ldcg(rq + 2);
    vupd = __ldcg(rq + 3);
  }
  const int vpc = vN - pv.window, vwlim = vN + 1 - pv.window;
  ArgMin bh{~0ull, -1}, bl{~0ull, -1}, bm{~0ull, -1};
  int xc = -1;
  float ic = 0.0f;
  for (int step = xb, it = 0; step < nsteps; step += nb, it++) {
    const int c0 = step * EC, c1 = min(nch, c0 + EC);
    if (it > 0) {                 // the rows of this step, after every thread is done with the last
      __syncthreads();
      if (threadIdx.x == 0) {
        const uint32_t bytes = (uint32_t)(c1 - c0) * a.lrow * 4u;
        mbar_expect_tx(bar, bytes);
        bulk_g2s(smem_u32(s_rows), a.logit + ((size_t)u * a.max_chunks + c0) * a.lrow, bytes, bar);
      }
    }
    // the positions of the block's next step, in flight during this one
    int vq[kPosRegs], vdq[kPosRegs / 4];
    float vsq[kPosRegs];
    if (step + nb < nsteps) load_positions<EC, MID>(pv, row_tab, paged, step + nb, nch, hc, vq, vsq, vdq);
    // one decision for the block, so that no thread is left at a barrier
    if (__syncthreads_or(!mbar_wait_bounded(bar, it & 1))) {
      if (threadIdx.x == 0 && atomicCAS(&pv.ctl->error, 0, DKV_ERR_TIMEOUT) == 0) pv.ctl->error_info = u;
      mbar_wait_bounded(bar, it & 1);
      return;
    }
    if (paged) {
      // four consecutive slots of one chunk per thread (pages hold whole
      // chunks, so the four share a page and their scores one 16-byte word):
      // S_j += 2^(max over queries of (l2 - lse2))
#pragma unroll
      for (int k = 0; k < EC * kChunk / 4 / kEpiThreads; k++) {
        const int x = k * kEpiThreads + threadIdx.x;
        const int lc = c0 + (x >> 2), j0 = 4 * (x & 3);
        if (lc >= c1) break;
        int s0, nt;
        const int tier = hc.tier(lc, s0, nt);
        s0 += j0;
        const int n = nt - s0;                    // valid slots among the four
        if (n <= 0) continue;
        const float* row = s_rows + (size_t)(lc - c0) * a.lrow;
        float4 mx = *reinterpret_cast<const float4*>(row + j0);
        mx.x -= lse[0]; mx.y -= lse[0]; mx.z -= lse[0]; mx.w -= lse[0];
#pragma unroll
        for (int qh = 1; qh < G; qh++) {
          const float4 v = *reinterpret_cast<const float4*>(row + qh * kChunk + j0);
          mx.x = fmaxf(mx.x, v.x - lse[qh]);
          mx.y = fmaxf(mx.y, v.y - lse[qh]);
          mx.z = fmaxf(mx.z, v.z - lse[qh]);
          mx.w = fmaxf(mx.w, v.w - lse[qh]);
        }
        const float4 old = make_float4(vs[4 * k], vs[4 * k + 1], vs[4 * k + 2], vs[4 * k + 3]);
        const int pid = vd[k];
        const TierGeom& tg = tier_geom<MID>(pv, tier);
        float* sp = reinterpret_cast<float*>(pv.page(pid) + tg.off[4]) + (s0 - tg.div(s0) * tg.t);
        const float4 nw = make_float4(old.x + fast_exp2(mx.x), old.y + fast_exp2(mx.y), old.z + fast_exp2(mx.z),
                                      old.w + fast_exp2(mx.w));
        if (n >= 4) {
          *reinterpret_cast<float4*>(sp) = nw;
        } else {
          sp[0] = nw.x;
          if (n > 1) sp[1] = nw.y;
          if (n > 2) sp[2] = nw.z;
        }
        if (victims) {
          victim_token(nw.x, vp[4 * k], s0, tier, vn0, vupd, vpc, vwlim, bh, bl, bm, xc, ic);
          if (n > 1) victim_token(nw.y, vp[4 * k + 1], s0 + 1, tier, vn0, vupd, vpc, vwlim, bh, bl, bm, xc, ic);
          if (n > 2) victim_token(nw.z, vp[4 * k + 2], s0 + 2, tier, vn0, vupd, vpc, vwlim, bh, bl, bm, xc, ic);
          if (n > 3) victim_token(nw.w, vp[4 * k + 3], s0 + 3, tier, vn0, vupd, vpc, vwlim, bh, bl, bm, xc, ic);
        }
      }
    } else {
#pragma unroll
      for (int k = 0; k < EC * kChunk / kEpiThreads; k++) {
        const int x = k * kEpiThreads + threadIdx.x;
        const int lc = c0 + x / kChunk, j = x % kChunk;
        if (lc >= c1) break;
        int slot, nt;
        const int tier = hc.tier(lc, slot, nt);
        slot += j;
        if (slot >= nt) continue;
        const float* row = s_rows + (size_t)(lc - c0) * a.lrow;
        float pm = 0.0f;
#pragma unroll
        for (int qh = 0; qh < G; qh++) pm = fmaxf(pm, fast_exp2(row[qh * kChunk + j] - lse[qh]));
        // chunked path: page from the table, old score from the page
        const TierGeom& tg = tier_geom<MID>(pv, tier);
        const int d = tg.div(slot);
        const int pid = __ldcg(row_tab + tier_entry<MID>(pv, tier, d));
        float* sp = reinterpret_cast<float*>(pv.page(pid) + tg.off[4]) + (slot - d * tg.t);
        const float ns = __ldcg(sp) + pm;
        *sp = ns;
        if (victims) victim_token(ns, vp[k], slot, tier, vn0, vupd, vpc, vwlim, bh, bl, bm, xc, ic);
      }
    }
#pragma unroll
    for (int e = 0; e < kPosRegs; e++) {
      vp[e] = vq[e];
      vs[e] = vsq[e];
    }
#pragma unroll
    for (int e = 0; e < kPosRegs / 4; e++) vd[e] = vdq[e];
  }
  if (!victims) return;
  // each warp leaves its share of the head's victim keys (one partial a
  // warp, no barrier); the next generation step reduces the head's partials
#pragma unroll
  for (int sft = 16; sft >= 1; sft >>= 1) {
    bh = shfl_amin(bh, sft);
    bl = shfl_amin(bl, sft);
    if (MID) bm = shfl_amin(bm, sft);
  }
  const unsigned has = __ballot_sync(0xffffffffu, xc >= 0);   // t_c is one slot of the head
  const int src = has ? __ffs(has) - 1 : 0;
  xc = __shfl_sync(0xffffffffu, xc, src);
  ic = __shfl_sync(0xffffffffu, ic, src);
  if (lane == 0)
    pv.vpart(a.layer, sa.slots[i], kvh)[xb * kEpiWarps + warp] =
        VictimPart{bh.key, bl.key, bm.key, bh.slot, bl.slot, bm.slot, xc, ic, vN, vupd, nb * kEpiWarps};
  if (xb == 0 && threadIdx.x == 0)         // the head's stamps, in their own array
    *pv.vst(a.layer, sa.slots[i], kvh) = make_int4(vN, vupd, nb * kEpiWarps, 0);
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

// The paged attention kernel for the pool's group size and tier count.
template <bool MID>
static cudaError_t launch_paged(Pool& P, const AttnArgs& a, const SlotArgs& sa, int w, dim3 grid, dim3 block,
                                int smem, cudaStream_t st) {
  if (w != kWarpsPerSm)
    return launch_dependent(k_attn_paged<kAttnWarps, 0, MID>, grid, block, (size_t)smem, st, P.pv, a, sa);
  if (P.pv.G == 4)
    return launch_dependent(k_attn_paged<kWarpsPerSm, 4, MID>, grid, block, (size_t)smem, st, P.pv, a, sa);
  if (P.pv.G == 8)
    return launch_dependent(k_attn_paged<kWarpsPerSm, 8, MID>, grid, block, (size_t)smem, st, P.pv, a, sa);
  return launch_dependent(k_attn_paged<kWarpsPerSm, 0, MID>, grid, block, (size_t)smem, st, P.pv, a, sa);
}

// The epilogue for group size G.
template <bool MID>
static cudaError_t launch_epi(cudaLaunchConfig_t& lc, int G, Pool& P, const AttnArgs& a, const SlotArgs& sa) {
  switch (G) {
    case 1: return cudaLaunchKernelEx(&lc, k_attn_epi<1, MID>, P.pv, a, sa);
    case 2: return cudaLaunchKernelEx(&lc, k_attn_epi<2, MID>, P.pv, a, sa);
    case 3: return cudaLaunchKernelEx(&lc, k_attn_epi<3, MID>, P.pv, a, sa);
    case 4: return cudaLaunchKernelEx(&lc, k_attn_epi<4, MID>, P.pv, a, sa);
    case 5: return cudaLaunchKernelEx(&lc, k_attn_epi<5, MID>, P.pv, a, sa);
    case 6: return cudaLaunchKernelEx(&lc, k_attn_epi<6, MID>, P.pv, a, sa);
    case 7: return cudaLaunchKernelEx(&lc, k_attn_epi<7, MID>, P.pv, a, sa);
    default: return cudaLaunchKernelEx(&lc, k_attn_epi<8, MID>, P.pv, a, sa);
  }
}

// Launch the attention kernel of the pool's page geometry, then the epilogue
// kernel (merge and score update) as its programmatic dependent, over the
// scratch that `a` points to.
static cudaError_t launch_kernels(Pool& P, AttnArgs a, const SlotArgs& sa, int max_tokens, cudaStream_t st) {
  const int n_units = sa.n * P.pv.hkv;
  const bool paged = P.pv.hi.t % kChunk == 0 && P.pv.lo.t % kChunk == 0;
  int smem, w;   // w: warps per CTA
  if (paged) {
    a.mseg = 0;
    a.maxp = 1;
    a.stage_bytes = std::max(P.pv.hi.off[4], P.pv.lo.off[4]);
    if (P.pv.mid_enabled) a.stage_bytes = std::max(a.stage_bytes, P.pv.mid.off[4]);
    // per warp its page ring with mbarriers and its descriptor table; the head prefix
    auto need = [&](int warps) { return warps * (kPageStages * (a.stage_bytes + 8) + 64 * 16) + 4 * (n_units + 1); };
    w = need(kWarpsPerSm) <= kMaxAttnSmem ? kWarpsPerSm : kAttnWarps;
    smem = need(w);
  } else {
    a.mseg = (4 * std::max(P.pv.hi.t, P.pv.lo.t) + 15) & ~15;
    a.maxp = std::max(pages_per_chunk(P.pv.hi.t), pages_per_chunk(P.pv.lo.t));
    a.stage_bytes = kOffMeta + 2 * a.maxp * a.mseg;
    w = kAttnWarps;
    smem = kAttnWarps * kStages * (a.stage_bytes + 8) + 4 * (n_units + 1);
  }
  if (smem > kMaxAttnSmem) return cudaErrorInvalidConfiguration;
  a.paged = paged ? 1 : 0;
  a.lrow = P.pv.G * kChunk;
  a.nwarps = P.sm_count * kWarpsPerSm;
  const dim3 grid(P.sm_count * (kWarpsPerSm / w)), block(32 * w);
  cudaError_t e;
  if (!paged)
    e = launch_dependent(k_attn_decode, grid, block, (size_t)smem, st, P.pv, a, sa);
  else if (P.pv.mid_enabled)
    e = launch_paged<true>(P, a, sa, w, grid, block, smem, st);
  else
    e = launch_paged<false>(P, a, sa, w, grid, block, smem, st);
  if (e != cudaSuccess) return e;
  // epilogue: merge and (with score updates) the new scores
  const int G = P.pv.G;
  const EpiSmem es(G, a.update != 0);
  unsigned gx;
  if (a.update) {
    // chunk steps of the call's longest head, at most one wave of blocks
    // (four per SM) over all heads
    const int call_chunks = (max_tokens + kChunk - 1) / kChunk + (P.pv.mid_enabled ? 2 : 1);
    const int steps = (call_chunks + epi_chunks(G) - 1) / epi_chunks(G);
    gx = (unsigned)std::max(1, std::min(steps, 4 * P.sm_count / std::max(1, n_units)));
  } else {
    gx = (unsigned)((G * kSlices + kEpiWarps - 1) / kEpiWarps);
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(gx, (unsigned)n_units);
  lc.blockDim = dim3(kEpiThreads);
  lc.dynamicSmemBytes = (size_t)es.total;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  e = P.pv.mid_enabled ? launch_epi<true>(lc, G, P, a, sa) : launch_epi<false>(lc, G, P, a, sa);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_attention(Pool& P, int layer, const SlotArgs& sa, int max_tokens, const __half* q,
                             float* out, int update_scores, cudaStream_t st) {
  AttnArgs a;
  a.q = q;
  a.out = out;
  a.part = P.sc.apart;
  a.logit = P.sc.alogit;
  a.lse2 = P.sc.alse;
  a.victims = 1;
  a.max_parts = P.sc.max_splits;
  a.max_chunks = P.sc.max_chunks;
  a.update = update_scores;
  a.layer = layer;
  return launch_kernels(P, a, sa, max_tokens, st);
}

// ---------------------------------------------------------------------------
// Allocation-free variant (dkv_decode_attention_static). The same kernels
// work in one fixed device array instead of the pool's scratch: the per-head
// lse2, the per-warp partials and, with score updates, the per-chunk rows of
// logits. The array is part of this library's device image; the CUDA driver
// reserves it when the module is loaded, so no call here allocates. Every
// call shares it and it keeps the last call's contents.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_attn_static_scratch[DKV_ATTN_STATIC_SCRATCH_BYTES];

namespace {
size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Regions of the array for one call, each 256-byte aligned: lse2 at 0, then
// partials, chunk rows. Strides are sized for the call's longest request, not
// the pool's maximum.
struct StaticLayout {
  size_t lse2, part, logit, total;
  int max_parts, max_chunks;
};

StaticLayout static_layout(int n_units, int G, int max_tokens, int update_scores, bool mid) {
  StaticLayout L;
  // a head's chunks: each tier's tokens rounded up to 16
  L.max_chunks = (max_tokens + kChunk - 1) / kChunk + (mid ? 2 : 1);
  L.max_parts = L.max_chunks / kMinChunks + 2;   // warps over one head (ranges >= kMinChunks)
  size_t off = 0;
  L.lse2 = off;
  off = round256(off + (size_t)n_units * G * sizeof(float));
  L.part = off;
  off = round256(off + (size_t)n_units * L.max_parts * part_stride(G) * sizeof(float));
  L.logit = off;
  if (update_scores) off += (size_t)n_units * L.max_chunks * G * kChunk * sizeof(float);
  L.total = off;
  return L;
}

}  // namespace

// Address of the array on the current device (call with the pool's device
// current). dkv_pool_create looks it up once and keeps it in the pool: a pool
// made after the device's context was reset holds the address in the new
// context.
cudaError_t static_scratch_address(void** base) {
  *base = nullptr;
  return cudaGetSymbolAddress(base, g_attn_static_scratch);
}

size_t attention_static_bytes(const Pool& P, int n_units, int max_tokens, int update_scores) {
  return static_layout(n_units, P.pv.G, max_tokens, update_scores, P.pv.mid_enabled != 0).total;
}

cudaError_t launch_attention_static(Pool& P, int layer, const SlotArgs& sa, int max_tokens, const __half* q,
                                    float* out, int update_scores, cudaStream_t st) {
  const int n_units = sa.n * P.pv.hkv;
  const StaticLayout L = static_layout(n_units, P.pv.G, max_tokens, update_scores, P.pv.mid_enabled != 0);
  if (L.total > DKV_ATTN_STATIC_SCRATCH_BYTES) return cudaErrorInvalidValue;
  uint8_t* base = static_cast<uint8_t*>(P.static_base);
  if (base == nullptr) return cudaErrorInvalidSymbol;
  AttnArgs a;
  a.q = q;
  a.out = out;
  a.lse2 = reinterpret_cast<float*>(base + L.lse2);
  a.part = reinterpret_cast<float*>(base + L.part);
  a.logit = reinterpret_cast<float*>(base + L.logit);
  a.max_parts = L.max_parts;
  a.max_chunks = L.max_chunks;
  a.victims = 0;                  // no victim keys: the next generation step scans
  a.update = update_scores;
  a.layer = layer;
  // Nothing in the array needs clearing: every value a call reads from it
  // (partials, chunk rows) is written earlier in the same call.
  return launch_kernels(P, a, sa, max_tokens, st);
}

template <bool MID>
static void attention_fns(std::vector<const void*>& fns) {
  fns.push_back(reinterpret_cast<const void*>(k_attn_paged<kWarpsPerSm, 4, MID>));
  fns.push_back(reinterpret_cast<const void*>(k_attn_paged<kWarpsPerSm, 8, MID>));
  fns.push_back(reinterpret_cast<const void*>(k_attn_paged<kWarpsPerSm, 0, MID>));
  fns.push_back(reinterpret_cast<const void*>(k_attn_paged<kAttnWarps, 0, MID>));
  fns.push_back(reinterpret_cast<const void*>(k_attn_epi<1, MID>));
  fns.push_back(reinterpret_cast<const void*>(k_attn_epi<2, MID>));
  fns.push_back(reinterpret_cast<const void*>(k_attn_epi<3, MID>));
  fns.push_back(reinterpret_cast<const void*>(k_attn_epi<4, MID>));
  fns.push_back(reinterpret_cast<const void*>(k_attn_epi<5, MID>));
  fns.push_back(reinterpret_cast<const void*>(k_attn_epi<6, MID>));
  fns.push_back(reinterpret_cast<const void*>(k_attn_epi<7, MID>));
  fns.push_back(reinterpret_cast<const void*>(k_attn_epi<8, MID>));
}

cudaError_t configure_attention() {
  std::vector<const void*> fns{reinterpret_cast<const void*>(k_attn_decode)};
  attention_fns<false>(fns);
  attention_fns<true>(fns);
  for (const void* f : fns) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxAttnSmem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dkv
