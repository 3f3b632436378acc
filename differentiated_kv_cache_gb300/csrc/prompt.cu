// prompt.cu — prompt-phase compaction kernels (DiffKV, compaction policy,
// prompt phase; memory management, prompt workflow, Figure 6).
//
//   k_prompt_given    tier and in-block rank from scores (caller-given or computed)
//   k_prompt_scatter  rank -> position map per (head, tier)
//   k_prompt_pack     quantize and pack surviving tokens into the granted pages
//
// Token scores from the observation queries (log-sum-exp pass, merge, score
// pass) run on the tensor cores in prompt_tc.cu, and k_prompt_given then
// takes the tiers and ranks from them; the allocation step between score and
// scatter (grant prefix sum, reclaim, table) is in alloc.cu.
#include "dkv_kernels.cuh"

namespace dkv {

// Tier of one prompt token and its rank among same-tier tokens of the block
// (block of kKeyBlock consecutive positions handled by 128 threads). A
// three-tier pool also splits off mid tokens (am: the head's alpha_m) and
// counts them in *bcm_out (MID).
template <bool MID>
__device__ __forceinline__ void classify_block(const PoolView& pv, float2 al, float am, int n0, int j, float s,
                                               int& tier, int& rank, int* s_cnt /*[3*4]*/, int2* bcnt_out,
                                               int* bcm_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  tier = kTierPrune;
  if (j < n0) {
    if (j >= n0 - pv.window) {
      tier = kTierHi;
    } else {
      const float imp = __fdiv_rn(s, (float)score_count(j, n0, 0));
      const float th_h = __fdiv_rn(al.x, (float)n0), th_l = __fdiv_rn(al.y, (float)n0);
      tier = MID ? classify3(imp, th_h, __fdiv_rn(am, (float)n0), th_l) : classify(imp, th_h, th_l, pv.lo_enabled);
    }
  }
  const unsigned bh = __ballot_sync(0xffffffffu, tier == kTierHi);
  const unsigned bl = __ballot_sync(0xffffffffu, tier == kTierLo);
  const unsigned bm = MID ? __ballot_sync(0xffffffffu, tier == kTierMid) : 0u;
  if (lane == 0) {
    s_cnt[warp] = __popc(bh);
    s_cnt[4 + warp] = __popc(bl);
    if (MID) s_cnt[8 + warp] = __popc(bm);
  }
  __syncthreads();
  int bh0 = 0, bl0 = 0, bm0 = 0;
  for (int w = 0; w < warp; w++) {
    bh0 += s_cnt[w];
    bl0 += s_cnt[4 + w];
    if (MID) bm0 += s_cnt[8 + w];
  }
  const unsigned below = (1u << lane) - 1u;
  rank = tier == kTierHi ? bh0 + __popc(bh & below)
                         : (tier == kTierLo ? bl0 + __popc(bl & below) : (tier == kTierMid ? bm0 + __popc(bm & below) : 0));
  if (tid == 0 && bcnt_out)
    *bcnt_out = make_int2(s_cnt[0] + s_cnt[1] + s_cnt[2] + s_cnt[3], s_cnt[4] + s_cnt[5] + s_cnt[6] + s_cnt[7]);
  if (MID && tid == 0) *bcm_out = s_cnt[8] + s_cnt[9] + s_cnt[10] + s_cnt[11];
}

// Tier from caller-given scores (score_in), same rule and ranks, against the
// thresholds of the token's head. MID: a three-tier pool.
template <bool MID>
__global__ void __launch_bounds__(128) k_prompt_given(PoolView pv, int layer, const float* __restrict__ score_in,
                                                       float* score_out, uint16_t* tokinfo, int2* bcnt, int* bcnt_m,
                                                       int nkb_cap) {
  if (pv.noop()) return;
  __shared__ int s_cnt[12];
  const int kb = blockIdx.x, kvh = blockIdx.y, i = blockIdx.z;
  const CallArgs* ca = pv.call;
  const int n0 = ca->lens[i];
  const int key0 = kb * kKeyBlock;
  if (key0 >= n0) return;
  const int j = key0 + threadIdx.x;
  const size_t tok = (size_t)(ca->tok0[i] + j) * pv.hkv + kvh;
  const float s = j < n0 ? score_in[tok] : 0.0f;
  int tier, rank;
  const size_t bx = ((size_t)i * pv.hkv + kvh) * nkb_cap + kb;
  classify_block<MID>(pv, pv.thresholds(layer, kvh), MID ? pv.alpha_m[(size_t)layer * pv.hkv + kvh] : 0.0f, n0, j,
                      s, tier, rank, s_cnt, bcnt + bx, bcnt_m + bx);
  if (j < n0) {
    if (score_out) score_out[tok] = s;
    tokinfo[tok] = (uint16_t)((rank << 2) | tier);
  }
}

// rank -> position map of a head's tier: map 0 lo, 1 hi, 2 mid
__device__ __forceinline__ int tier_map(int tier) { return tier == kTierHi ? 1 : (tier == kTierLo ? 0 : 2); }

// rank2pos[unit][map][rank] = position, rank = block base + in-block rank.
__global__ void __launch_bounds__(128) k_prompt_scatter(PoolView pv, const uint16_t* __restrict__ tokinfo,
                                                         const int2* __restrict__ bbase,
                                                         const int* __restrict__ bbase_m, int* rank2pos,
                                                         int nkb_cap) {
  if (pv.noop()) return;
  const int kb = blockIdx.x, kvh = blockIdx.y, i = blockIdx.z;
  const CallArgs* ca = pv.call;
  const int n0 = ca->lens[i];
  const int j = kb * kKeyBlock + threadIdx.x;
  if (j >= n0) return;
  const size_t unit = (size_t)i * pv.hkv + kvh;
  const uint16_t info = tokinfo[(size_t)(ca->tok0[i] + j) * pv.hkv + kvh];
  const int tier = info & 3;
  if (tier == kTierPrune) return;
  int base;
  if (tier == kTierMid) {
    base = bbase_m[unit * nkb_cap + kb];
  } else {
    const int2 b2 = bbase[unit * nkb_cap + kb];
    base = tier == kTierHi ? b2.x : b2.y;
  }
  const int rank = base + (info >> 2);
  rank2pos[(unit * (pv.mid_enabled ? 3 : 2) + tier_map(tier)) * pv.max_seq + rank] = j;
}

// ---------------------------------------------------------------------------
// a4: quantize + pack (hi: K8V4, lo: K4V2). A warp handles groups of 8
// consecutive ranks of one head's tier: 4 lanes per token, 32 features per
// lane. A group fills whole value rows (4 pair-rows hi, 2 quad-rows lo); the
// value words are assembled in shared memory and written as full 128-byte
// rows. The codes follow qcode (the oracle's arithmetic); a zero scale has
// inv = 0, which gives code 0 without a branch.
// ---------------------------------------------------------------------------
constexpr int kPackTok = 8;      // tokens per group

// Code arithmetic of qcode, taken apart: t = (x - z) * inv for a pair in
// packed fp32, then round to nearest even into s32 (saturating; NaN gives 0),
// and the clamp to [0, 2^B - 1] happens in the packing instruction, which
// shifts the word built so far up and inserts two saturated fields:
//   cvt.pack.sat.uB.s32.b32 d, a, b, c:  d = (c << 2B) | (sat(a) << B) | sat(b)
__device__ __forceinline__ void qt2(float x0, float x1, const QParams& q, int& r0, int& r1) {
  const uint64_t t = mul_f32x2(sub_f32x2(f32x2(x0, x1), f32x2(q.z, q.z)), f32x2(q.inv, q.inv));
  asm("cvt.rni.s32.f32 %0, %1;\n" : "=r"(r0) : "f"(__uint_as_float((uint32_t)t)));
  asm("cvt.rni.s32.f32 %0, %1;\n" : "=r"(r1) : "f"(__uint_as_float((uint32_t)(t >> 32))));
}
template <int B>
__device__ __forceinline__ uint32_t pack_sat(int a, int b, uint32_t c) {
  uint32_t d;
  if (B == 8) asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  if (B == 4) asm("cvt.pack.sat.u4.s32.b32 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  if (B == 2) asm("cvt.pack.sat.u2.s32.b32 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// The group of 8 consecutive ranks r0 .. r0+7 of one head's tier. Lane
// (e, q) holds token e's K and V features 32q .. 32q+31 in kv (4 uint4 of K,
// then 4 of V) and its position j (-1 past the tier's count); grant: the
// head's granted page IDs; s_vw: the warp's [token][value word] scratch.
// TIER: hi (K8V4, pages from the grant's left), lo (K4V2, from its right) or
// mid (K8V2, from grant entry mbase on: the pages after the hi ones).
template <int TIER>
__device__ __forceinline__ void pack_group(const PoolView& pv, const uint4 (&kv)[8], int j, int r0, int count,
                                           int gcnt, int mbase, const int* __restrict__ grant,
                                           const float* __restrict__ score, size_t tok_base, int kvh,
                                           uint32_t (*s_vw)[32]) {
  constexpr bool HI = TIER == kTierHi, LOW = TIER == kTierLo;
  constexpr int KB = LOW ? 4 : 8, VB = HI ? 4 : 2, GSZ = 8 / VB;   // GSZ: tokens per value row
  const TierGeom& tg = HI ? pv.hi : (LOW ? pv.lo : pv.mid);
  const int lane = threadIdx.x & 31, e = lane >> 2, q = lane & 3;   // token e of the 8, features 32q..32q+31
  // bit offset of this token's slot inside a value word
  const int slot_e = e % GSZ;
  const int eb = VB == 4 ? 16 * slot_e : 16 * (slot_e & 1) + 2 * (slot_e >> 1);
  const int r = r0 + e;
  const bool valid = r < count;
  const __half2* kh = reinterpret_cast<const __half2*>(&kv[0]);   // 16 pairs
  const __half2* vh = reinterpret_cast<const __half2*>(&kv[4]);
  float kmn, kmx, vmn, vmx;
  {
    __half2 kmn2 = kh[0], kmx2 = kh[0], vmn2 = vh[0], vmx2 = vh[0];
#pragma unroll
    for (int y = 1; y < 16; y++) {   // min / max of fp16 values are exact
      kmn2 = __hmin2(kmn2, kh[y]);
      kmx2 = __hmax2(kmx2, kh[y]);
      vmn2 = __hmin2(vmn2, vh[y]);
      vmx2 = __hmax2(vmx2, vh[y]);
    }
    kmn = fminf(__low2float(kmn2), __high2float(kmn2));
    kmx = fmaxf(__low2float(kmx2), __high2float(kmx2));
    vmn = fminf(__low2float(vmn2), __high2float(vmn2));
    vmx = fmaxf(__low2float(vmx2), __high2float(vmx2));
  }
  // every lane takes part in the token reductions; invalid lanes hold zeros
#pragma unroll
  for (int sh = 1; sh <= 2; sh <<= 1) {
    kmn = fminf(kmn, __shfl_xor_sync(0xffffffffu, kmn, sh, 4));
    kmx = fmaxf(kmx, __shfl_xor_sync(0xffffffffu, kmx, sh, 4));
    vmn = fminf(vmn, __shfl_xor_sync(0xffffffffu, vmn, sh, 4));
    vmx = fmaxf(vmx, __shfl_xor_sync(0xffffffffu, vmx, sh, 4));
  }
  const QParams kq = qparams(kmn, kmx, KB), vq = qparams(vmn, vmx, VB);
  // the token's bits of value words 8q .. 8q+7 (features 4w .. 4w+3)
  __syncwarp();                              // the previous group's value rows are written
#pragma unroll
  for (int w = 0; w < 8; w++) {
    // the token's codes of features 4w .. 4w+3 at bits 4i of its 16-bit field
    const float2 a = __half22float2(vh[2 * w]), b = __half22float2(vh[2 * w + 1]);
    int c0, c1, c2, c3;
    qt2(a.x, a.y, vq, c0, c1);
    qt2(b.x, b.y, vq, c2, c3);
    uint32_t f;
    if (VB == 4) {
      f = pack_sat<4>(c1, c0, pack_sat<4>(c3, c2, 0u));
    } else {                               // 2-bit codes 4 bits apart (zero between)
      f = pack_sat<2>(0, c0, pack_sat<2>(0, c1, pack_sat<2>(0, c2, pack_sat<2>(0, c3, 0u))));
    }
    s_vw[e][8 * q + w] = valid ? f << eb : 0u;
  }
  if (valid) {
    // page and slot of rank r: hi from the left of the grant, lo from the
    // right, mid from mbase on
    const int pidx = HI ? tg.div(r) : (LOW ? gcnt - 1 - tg.div(r) : mbase + tg.div(r));
    const int slot = r - tg.div(r) * tg.t;
    uint8_t* page = pv.page(grant[pidx]);
    uint8_t* krow = page + tg.off[0] + slot * tg.kbytes;
    if (KB == 8) {
      uint32_t w[8];
#pragma unroll
      for (int y = 0; y < 8; y++) {             // bytes 4y .. 4y+3
        const float2 a = __half22float2(kh[2 * y]), b = __half22float2(kh[2 * y + 1]);
        int c0, c1, c2, c3;
        qt2(a.x, a.y, kq, c0, c1);
        qt2(b.x, b.y, kq, c2, c3);
        w[y] = pack_sat<8>(c1, c0, pack_sat<8>(c3, c2, 0u));
      }
      uint4* dst = reinterpret_cast<uint4*>(krow + 32 * q);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
      uint32_t w[4];
#pragma unroll
      for (int y = 0; y < 4; y++) {             // bytes 4y .. 4y+3: features 8y .. 8y+7
        uint32_t acc = 0u;
#pragma unroll
        for (int z = 3; z >= 0; z--) {          // byte z: feature 2z low nibble, 2z + 1 high
          const float2 a = __half22float2(kh[4 * y + z]);
          int c0, c1;
          qt2(a.x, a.y, kq, c0, c1);
          acc = pack_sat<4>(c1, c0, acc);
        }
        w[y] = acc;
      }
      *reinterpret_cast<uint4*>(krow + 16 * q) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (q == 0) {
      const size_t tok = (tok_base + j) * pv.hkv + kvh;
      *reinterpret_cast<uint32_t*>(page + tg.off[2] + 4 * slot) = (uint32_t)kq.sh | ((uint32_t)kq.zh << 16);
      *reinterpret_cast<uint32_t*>(page + tg.off[3] + 4 * slot) = (uint32_t)vq.sh | ((uint32_t)vq.zh << 16);
      *reinterpret_cast<float*>(page + tg.off[4] + 4 * slot) = score[tok];
      *reinterpret_cast<int*>(page + tg.off[5] + 4 * slot) = j;
    }
  }
  __syncwarp();
  // value rows: GSZ tokens each (4 pair-rows hi, 2 quad-rows lo)
#pragma unroll
  for (int row = 0; row < kPackTok / GSZ; row++) {
    const int rfirst = r0 + row * GSZ;
    if (rfirst >= count) break;
    const int pidx = HI ? tg.div(rfirst) : (LOW ? gcnt - 1 - tg.div(rfirst) : mbase + tg.div(rfirst));
    const int slot0 = rfirst - tg.div(rfirst) * tg.t;
    uint8_t* page = pv.page(grant[pidx]);
    uint32_t word = 0;
#pragma unroll
    for (int ee = 0; ee < GSZ; ee++) word |= s_vw[row * GSZ + ee][lane];
    *reinterpret_cast<uint32_t*>(page + tg.off[1] + (slot0 / GSZ) * 128 + 4 * lane) = word;
  }
}

// One persistent grid over both tiers of every head of the call: the groups
// are numbered head by head (the head's hi groups, then its lo groups) and
// warp w of the grid takes groups w, w + W, w + 2W, ... (W warps in all), so
// that every warp streams one long sequence with its loads ahead of the math:
// the positions of the group after next and the K/V rows of the next group
// are in flight while a group is quantized and stored.
// A three-tier pool's heads (MID) also have mid groups (after their lo
// groups); unit_mid holds each head's mid token count.
template <bool MID>
__global__ void __launch_bounds__(256, 2) k_prompt_pack(PoolView pv, const __half* __restrict__ k,
                                                         const __half* __restrict__ v,
                                                         const float* __restrict__ score,
                                                         const int* __restrict__ rank2pos,
                                                         const int4* __restrict__ unit_info,
                                                         const int* __restrict__ unit_mid,
                                                         const int* __restrict__ grant_ids, int grant_cap) {
  if (pv.noop()) return;
  extern __shared__ int s_pref[];              // [n_units + 1] first group of each head
  __shared__ uint32_t s_vw[8][kPackTok][32];   // [warp][token][value word] code bits of the token
  __shared__ int s_warp[8];
  const CallArgs* ca = pv.call;
  const int hkv = pv.hkv, n_units = ca->n_req * hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, e = lane >> 2, q = lane & 3;
  {
    // exclusive prefix over the heads of their group counts (a contiguous run of heads per thread)
    const int per = (n_units + blockDim.x - 1) / blockDim.x;
    const int u0 = min(n_units, (int)threadIdx.x * per), u1 = min(n_units, u0 + per);
    int sum = 0;
    for (int u = u0; u < u1; u++) {
      const int4 ui = unit_info[u];
      sum += (ui.y + kPackTok - 1) / kPackTok + (ui.z + kPackTok - 1) / kPackTok;
      if (MID) sum += (unit_mid[u] + kPackTok - 1) / kPackTok;
    }
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
      s_pref[u] = run;
      const int4 ui = unit_info[u];
      run += (ui.y + kPackTok - 1) / kPackTok + (ui.z + kPackTok - 1) / kPackTok;
      if (MID) run += (unit_mid[u] + kPackTok - 1) / kPackTok;
    }
    if (threadIdx.x == blockDim.x - 1) s_pref[n_units] = run;
    __syncthreads();
  }
  const int total = s_pref[n_units];
  const int W = gridDim.x * 8;
  struct Grp {
    int unit, r0, count, gcnt, tier, mbase;
  };
  constexpr int nmaps = MID ? 3 : 2;
  auto describe = [&](int x, Grp& d) {
    if (x >= total) return false;
    int lo = 0, hi = n_units - 1;              // last head with s_pref <= x
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pref[mid] <= x) lo = mid; else hi = mid - 1;
    }
    const int4 ui = unit_info[lo];
    const int gh = (ui.y + kPackTok - 1) / kPackTok, gl = (ui.z + kPackTok - 1) / kPackTok;
    const int off = x - s_pref[lo];
    d.unit = lo;
    d.tier = off < gh ? kTierHi : (!MID || off < gh + gl ? kTierLo : kTierMid);
    d.r0 = kPackTok * (off < gh ? off : (!MID || off < gh + gl ? off - gh : off - gh - gl));
    d.count = d.tier == kTierHi ? ui.y : (d.tier == kTierLo ? ui.z : unit_mid[lo]);
    d.gcnt = ui.x;
    d.mbase = MID ? pv.hi.div(ui.y + pv.hi.t - 1) : 0;   // mid pages follow the head's hi pages in its grant
    return true;
  };
  auto pos_of = [&](bool has, const Grp& d) {
    if (!has) return -1;
    const int r = d.r0 + e;
    const int map = d.tier == kTierHi ? 1 : (d.tier == kTierLo ? 0 : 2);
    return r < d.count ? __ldg(rank2pos + ((size_t)d.unit * nmaps + map) * pv.max_seq + r) : -1;
  };
  auto load_kv = [&](const Grp& d, int j, uint4 (&kv)[8]) {
    if (j >= 0) {
      const size_t tok = (size_t)(ca->tok0[d.unit / hkv] + j) * hkv + d.unit % hkv;
      const uint4* kp = reinterpret_cast<const uint4*>(k + tok * kD + q * 32);
      const uint4* vp = reinterpret_cast<const uint4*>(v + tok * kD + q * 32);
#pragma unroll
      for (int y = 0; y < 4; y++) {
        kv[y] = __ldg(kp + y);
        kv[4 + y] = __ldg(vp + y);
      }
    } else {
#pragma unroll
      for (int y = 0; y < 8; y++) kv[y] = make_uint4(0, 0, 0, 0);
    }
  };
  int x = blockIdx.x * 8 + warp;
  Grp dc, dn, da;
  bool hc = describe(x, dc), hn = describe(x + W, dn);
  int jc = pos_of(hc, dc), jn = pos_of(hn, dn);
  uint4 kvc[8], kvn[8];
  if (hc) load_kv(dc, jc, kvc);
  while (hc) {
    if (hn) load_kv(dn, jn, kvn);
    const bool ha = describe(x + 2 * W, da);
    const int ja = pos_of(ha, da);
    const int i = dc.unit / hkv, kvh = dc.unit % hkv;
    const int* grant = grant_ids + (size_t)dc.unit * grant_cap;
    if (dc.tier == kTierHi)
      pack_group<kTierHi>(pv, kvc, jc, dc.r0, dc.count, dc.gcnt, 0, grant, score, (size_t)ca->tok0[i], kvh,
                          s_vw[warp]);
    else if (dc.tier == kTierLo)
      pack_group<kTierLo>(pv, kvc, jc, dc.r0, dc.count, dc.gcnt, 0, grant, score, (size_t)ca->tok0[i], kvh,
                          s_vw[warp]);
    else if (MID)
      pack_group<kTierMid>(pv, kvc, jc, dc.r0, dc.count, dc.gcnt, dc.mbase, grant, score, (size_t)ca->tok0[i], kvh,
                           s_vw[warp]);
    dc = dn;
    hc = hn;
    jc = jn;
    dn = da;
    hn = ha;
    jn = ja;
#pragma unroll
    for (int y = 0; y < 8; y++) kvc[y] = kvn[y];
    x += W;
  }
}

// ---------------------------------------------------------------------------
cudaError_t launch_prompt_plan(Pool& P, int layer, int n_req, cudaStream_t st);
cudaError_t configure_attention();
cudaError_t configure_alloc();
cudaError_t configure_prompt_tc();
cudaError_t configure_prefill();
cudaError_t launch_scoring_tc(Pool& P, const __half* k, const __half* q_obs, const float* lse_obs, long long n_tok,
                              int n_req, float* score_out, cudaStream_t st);

cudaError_t configure_kernels() {
  cudaError_t e;
  if ((e = configure_prompt_tc()) != cudaSuccess) return e;
  if ((e = configure_alloc()) != cudaSuccess) return e;
  if ((e = configure_prefill()) != cudaSuccess) return e;
  // the pack kernel keeps one int per head of the call in shared memory
  if ((e = cudaFuncSetAttribute(k_prompt_pack<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_prompt_pack<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024)) !=
      cudaSuccess)
    return e;
  return configure_attention();
}

cudaError_t launch_prompt(Pool& P, int layer, int n_req, int max_len, long long n_tok, const __half* k,
                          const __half* v, const __half* q_obs, const float* lse_obs, const float* scores_in,
                          float* scores_out, cudaStream_t st) {
  const Scratch& s = P.sc;
  const int nkb = (max_len + kKeyBlock - 1) / kKeyBlock;
  const dim3 grid(nkb, P.pv.hkv, n_req);
  cudaError_t e = cudaSuccess;
  const float* score_src;
  if (scores_in) {
    if (P.pv.mid_enabled)
      k_prompt_given<true><<<grid, 128, 0, st>>>(P.pv, layer, scores_in, scores_out, s.tokinfo, s.bcnt, s.bcnt_m,
                                                 s.nkb_cap);
    else
      k_prompt_given<false><<<grid, 128, 0, st>>>(P.pv, layer, scores_in, scores_out, s.tokinfo, s.bcnt, s.bcnt_m,
                                                  s.nkb_cap);
    e = cudaGetLastError();
    score_src = scores_in;
  } else {
    float* so = scores_out ? scores_out : s.score;
    e = launch_scoring_tc(P, k, q_obs, lse_obs, n_tok, n_req, so, st);
    if (e == cudaSuccess) {      // tiers and in-block ranks from the scores
      if (P.pv.mid_enabled)
        k_prompt_given<true><<<grid, 128, 0, st>>>(P.pv, layer, so, nullptr, s.tokinfo, s.bcnt, s.bcnt_m, s.nkb_cap);
      else
        k_prompt_given<false><<<grid, 128, 0, st>>>(P.pv, layer, so, nullptr, s.tokinfo, s.bcnt, s.bcnt_m,
                                                    s.nkb_cap);
      e = cudaGetLastError();
    }
    score_src = so;
  }
  if (e != cudaSuccess) return e;
  if ((e = launch_prompt_plan(P, layer, n_req, st)) != cudaSuccess) return e;
  k_prompt_scatter<<<grid, 128, 0, st>>>(P.pv, s.tokinfo, s.bbase, s.bbase_m, s.rank2pos, s.nkb_cap);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t pref = sizeof(int) * ((size_t)n_req * P.pv.hkv + 1);
  if (P.pv.mid_enabled)
    k_prompt_pack<true><<<2 * P.sm_count, 256, pref, st>>>(P.pv, k, v, score_src, s.rank2pos, s.unit_info,
                                                           s.unit_mid, s.grant_ids, s.grant_cap);
  else
    k_prompt_pack<false><<<2 * P.sm_count, 256, pref, st>>>(P.pv, k, v, score_src, s.rank2pos, s.unit_info,
                                                            s.unit_mid, s.grant_ids, s.grant_cap);
  return cudaGetLastError();
}

}  // namespace dkv
