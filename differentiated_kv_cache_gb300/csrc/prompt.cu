// prompt.cu — prompt-phase compaction kernels (DiffKV, compaction policy,
// prompt phase; memory management, prompt workflow, Figure 6).
//
//   k_prompt_given    tier from caller-given scores
//   k_prompt_scatter  rank -> position map per (head, tier)
//   k_prompt_pack     quantize and pack surviving tokens into the granted pages
//
// Token scores from the observation queries (log-sum-exp pass, merge, score
// pass) run on the tensor cores in prompt_tc.cu; the allocation step between
// score and scatter (grant prefix sum, reclaim, table) is in alloc.cu.
#include "dkv_kernels.cuh"

namespace dkv {

// Tier of one prompt token and its rank among same-tier tokens of the block
// (block of kKeyBlock consecutive positions handled by 128 threads).
__device__ __forceinline__ void classify_block(const PoolView& pv, int n0, int j, float s, int& tier,
                                               int& rank, int* s_cnt /*[2*4]*/, int2* bcnt_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  tier = kTierPrune;
  if (j < n0) {
    if (j >= n0 - pv.window) {
      tier = kTierHi;
    } else {
      const float imp = __fdiv_rn(s, (float)score_count(j, n0, 0));
      tier = classify(imp, __fdiv_rn(pv.alpha_h, (float)n0), __fdiv_rn(pv.alpha_l, (float)n0), pv.lo_enabled);
    }
  }
  const unsigned bh = __ballot_sync(0xffffffffu, tier == kTierHi);
  const unsigned bl = __ballot_sync(0xffffffffu, tier == kTierLo);
  if (lane == 0) { s_cnt[warp] = __popc(bh); s_cnt[4 + warp] = __popc(bl); }
  __syncthreads();
  int bh0 = 0, bl0 = 0;
  for (int w = 0; w < warp; w++) { bh0 += s_cnt[w]; bl0 += s_cnt[4 + w]; }
  const unsigned below = (1u << lane) - 1u;
  rank = tier == kTierHi ? bh0 + __popc(bh & below) : (tier == kTierLo ? bl0 + __popc(bl & below) : 0);
  if (tid == 0 && bcnt_out)
    *bcnt_out = make_int2(s_cnt[0] + s_cnt[1] + s_cnt[2] + s_cnt[3], s_cnt[4] + s_cnt[5] + s_cnt[6] + s_cnt[7]);
}

// Tier from caller-given scores (score_in), same rule and ranks.
__global__ void __launch_bounds__(128) k_prompt_given(PoolView pv, const float* __restrict__ score_in,
                                                       float* score_out, uint16_t* tokinfo, int2* bcnt,
                                                       int nkb_cap) {
  if (pv.noop()) return;
  __shared__ int s_cnt[8];
  const int kb = blockIdx.x, kvh = blockIdx.y, i = blockIdx.z;
  const CallArgs* ca = pv.call;
  const int n0 = ca->lens[i];
  const int key0 = kb * kKeyBlock;
  if (key0 >= n0) return;
  const int j = key0 + threadIdx.x;
  const size_t tok = (size_t)(ca->tok0[i] + j) * pv.hkv + kvh;
  const float s = j < n0 ? score_in[tok] : 0.0f;
  int tier, rank;
  classify_block(pv, n0, j, s, tier, rank, s_cnt, bcnt + ((size_t)i * pv.hkv + kvh) * nkb_cap + kb);
  if (j < n0) {
    if (score_out) score_out[tok] = s;
    tokinfo[tok] = (uint16_t)((rank << 2) | tier);
  }
}

// rank2pos[unit][tier][rank] = position, rank = block base + in-block rank.
__global__ void __launch_bounds__(128) k_prompt_scatter(PoolView pv, const uint16_t* __restrict__ tokinfo,
                                                         const int2* __restrict__ bbase, int* rank2pos,
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
  const int2 base = bbase[unit * nkb_cap + kb];
  const int rank = (tier == kTierHi ? base.x : base.y) + (info >> 2);
  rank2pos[(unit * 2 + (tier == kTierHi ? 1 : 0)) * pv.max_seq + rank] = j;
}

// ---------------------------------------------------------------------------
// a4: quantize + pack. A warp handles groups of 4 consecutive ranks of one
// (head, tier): 8 lanes per token, 16 features per lane. A group fills two
// whole value pair-rows (hi) or one value quad-row (lo); the value words are
// assembled in shared memory and written as full 128-byte rows. Each warp
// takes kPackGroups groups in turn and keeps the loads ahead of the math: the
// positions of the group after next and the K/V rows of the next group are
// in flight while a group is quantized and stored.
// ---------------------------------------------------------------------------
constexpr int kPackGroups = 4;

__global__ void __launch_bounds__(256) k_prompt_pack(PoolView pv, const __half* __restrict__ k,
                                                      const __half* __restrict__ v,
                                                      const float* __restrict__ score,
                                                      const int* __restrict__ rank2pos,
                                                      const int4* __restrict__ unit_info,
                                                      const int* __restrict__ grant_ids, int grant_cap) {
  if (pv.noop()) return;
  __shared__ uint32_t s_vw[8][4][32];     // [warp][token][value word] code bits of the token
  const int unit = blockIdx.y, tier = blockIdx.z ? kTierHi : kTierLo;
  const int i = unit / pv.hkv, kvh = unit % pv.hkv;
  const int4 ui = unit_info[unit];        // grant pages, hi count, lo count, -
  const int count = tier == kTierHi ? ui.y : ui.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // group x of this warp starts at rank base + 32 x
  const int base = (blockIdx.x * kPackGroups * 8 + warp) * 4;
  if (base >= count) return;
  const TierGeom& tg = tier == kTierHi ? pv.hi : pv.lo;
  const int kbits = tier == kTierHi ? 8 : 4, vbits = tier == kTierHi ? 4 : 2;
  const int e = lane >> 3, q = lane & 7;  // token e of the 4, features 16q..16q+15
  const CallArgs* ca = pv.call;
  const int* r2p = rank2pos + ((size_t)unit * 2 + (tier == kTierHi ? 1 : 0)) * pv.max_seq;
  const size_t tok_base = (size_t)ca->tok0[i];
  const int gcnt = ui.x;
  auto pos_of = [&](int x) { const int r = base + 32 * x + e; return r < count ? __ldg(r2p + r) : -1; };
  auto load_kv = [&](int j, uint4 (&kv)[4]) {
    if (j >= 0) {
      const size_t tok = (tok_base + j) * pv.hkv + kvh;
      const uint4* kp = reinterpret_cast<const uint4*>(k + tok * kD + q * 16);
      const uint4* vp = reinterpret_cast<const uint4*>(v + tok * kD + q * 16);
      kv[0] = __ldg(kp); kv[1] = __ldg(kp + 1); kv[2] = __ldg(vp); kv[3] = __ldg(vp + 1);
    } else {
      kv[0] = kv[1] = kv[2] = kv[3] = make_uint4(0, 0, 0, 0);
    }
  };
  int j_cur = pos_of(0), j_next = pos_of(1);
  uint4 kv_cur[4], kv_next[4];
  load_kv(j_cur, kv_cur);
  for (int x = 0; x < kPackGroups; x++) {
    const int r0 = base + 32 * x;
    if (r0 >= count) break;
    int j_after = -1;
    if (x + 1 < kPackGroups) load_kv(j_next, kv_next);
    if (x + 2 < kPackGroups) j_after = pos_of(x + 2);
    const int r = r0 + e;
    const bool valid = r < count;
    const int j = j_cur;
    float kx[16], vx[16];
    float kmn, kmx, vmn, vmx;
    {
      const __half2* kh = reinterpret_cast<const __half2*>(&kv_cur[0]);   // 8 pairs: kv_cur[0..1]
      const __half2* vh = reinterpret_cast<const __half2*>(&kv_cur[2]);
      __half2 kmn2 = kh[0], kmx2 = kh[0], vmn2 = vh[0], vmx2 = vh[0];
#pragma unroll
      for (int y = 1; y < 8; y++) {   // min / max of fp16 values are exact
        kmn2 = __hmin2(kmn2, kh[y]); kmx2 = __hmax2(kmx2, kh[y]);
        vmn2 = __hmin2(vmn2, vh[y]); vmx2 = __hmax2(vmx2, vh[y]);
      }
      kmn = fminf(__low2float(kmn2), __high2float(kmn2));
      kmx = fmaxf(__low2float(kmx2), __high2float(kmx2));
      vmn = fminf(__low2float(vmn2), __high2float(vmn2));
      vmx = fmaxf(__low2float(vmx2), __high2float(vmx2));
#pragma unroll
      for (int y = 0; y < 8; y++) {
        const float2 kf = __half22float2(kh[y]), vf = __half22float2(vh[y]);
        kx[2 * y] = kf.x; kx[2 * y + 1] = kf.y;
        vx[2 * y] = vf.x; vx[2 * y + 1] = vf.y;
      }
    }
    // every lane takes part in the group reductions; invalid lanes hold zeros
#pragma unroll
    for (int sh = 1; sh <= 4; sh <<= 1) {
      kmn = fminf(kmn, __shfl_xor_sync(0xffffffffu, kmn, sh, 8));
      kmx = fmaxf(kmx, __shfl_xor_sync(0xffffffffu, kmx, sh, 8));
      vmn = fminf(vmn, __shfl_xor_sync(0xffffffffu, vmn, sh, 8));
      vmx = fmaxf(vmx, __shfl_xor_sync(0xffffffffu, vmx, sh, 8));
    }
    const QParams kq = qparams(kmn, kmx, kbits), vq = qparams(vmn, vmx, vbits);
    // the token's bits of value words 4q .. 4q+3 (feature 4w+i, slot e of the row)
    const int gsz = 8 / vbits;
    const int eb = vbits == 4 ? 16 * (e % 2) : 16 * (e & 1) + 2 * (e >> 1);
    uint32_t vw[4];
#pragma unroll
    for (int w = 0; w < 4; w++) {
      uint32_t c0, c1, c2, c3;
      qcode2(vx[4 * w], vx[4 * w + 1], vq, vbits, c0, c1);
      qcode2(vx[4 * w + 2], vx[4 * w + 3], vq, vbits, c2, c3);
      vw[w] = valid ? (c0 | (c1 << 4) | (c2 << 8) | (c3 << 12)) << eb : 0u;
    }
    __syncwarp();                        // the previous group's value rows are written
#pragma unroll
    for (int w = 0; w < 4; w++) s_vw[warp][e][4 * q + w] = vw[w];
    if (valid) {
      // page and slot of rank r: hi from the left of the grant, lo from the right
      const int pidx = tier == kTierHi ? r / tg.t : gcnt - 1 - r / tg.t;
      const int slot = r % tg.t;
      uint8_t* page = pv.page(grant_ids[(size_t)unit * grant_cap + pidx]);
      uint8_t* krow = page + tg.off[0] + slot * tg.kbytes;
      if (kbits == 8) {
        uint32_t w[4];
#pragma unroll
        for (int y = 0; y < 4; y++) {
          uint32_t c0, c1, c2, c3;
          qcode2(kx[4 * y], kx[4 * y + 1], kq, 8, c0, c1);
          qcode2(kx[4 * y + 2], kx[4 * y + 3], kq, 8, c2, c3);
          w[y] = __byte_perm(c0 | (c2 << 16), c1 | (c3 << 16), 0x6240);
        }
        *reinterpret_cast<uint4*>(krow + 16 * q) = make_uint4(w[0], w[1], w[2], w[3]);
      } else {
        uint32_t w[2];
#pragma unroll
        for (int y = 0; y < 2; y++) {
          uint32_t acc = 0;
#pragma unroll
          for (int z = 0; z < 8; z += 2) {
            uint32_t c0, c1;
            qcode2(kx[8 * y + z], kx[8 * y + z + 1], kq, 4, c0, c1);
            acc |= (c0 | (c1 << 4)) << (4 * z);
          }
          w[y] = acc;
        }
        *reinterpret_cast<uint2*>(krow + 8 * q) = make_uint2(w[0], w[1]);
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
    // value rows: hi = 2 pair-rows (tokens 0,1 and 2,3), lo = 1 quad-row
    const int nrows = 4 / gsz;
    for (int row = 0; row < nrows; row++) {
      const int rfirst = r0 + row * gsz;
      if (rfirst >= count) break;
      const int pidx = tier == kTierHi ? rfirst / tg.t : gcnt - 1 - rfirst / tg.t;
      const int slot0 = rfirst % tg.t;
      uint8_t* page = pv.page(grant_ids[(size_t)unit * grant_cap + pidx]);
      uint32_t word = 0;
      for (int ee = 0; ee < gsz; ee++) word |= s_vw[warp][row * gsz + ee][lane];
      *reinterpret_cast<uint32_t*>(page + tg.off[1] + (slot0 / gsz) * 128 + 4 * lane) = word;
    }
    j_cur = j_next;
    j_next = j_after;
#pragma unroll
    for (int y = 0; y < 4; y++) kv_cur[y] = kv_next[y];
  }
}

// ---------------------------------------------------------------------------
cudaError_t launch_prompt_plan(Pool& P, int layer, int n_req, cudaStream_t st);
cudaError_t configure_attention();
cudaError_t configure_alloc();
cudaError_t configure_prompt_tc();
cudaError_t launch_scoring_tc(Pool& P, const __half* k, const __half* q_obs, long long n_tok, int n_req,
                              float* score_out, cudaStream_t st);

cudaError_t configure_kernels() {
  cudaError_t e;
  if ((e = configure_prompt_tc()) != cudaSuccess) return e;
  if ((e = configure_alloc()) != cudaSuccess) return e;
  return configure_attention();
}

cudaError_t launch_prompt(Pool& P, int layer, int n_req, int max_len, long long n_tok, const __half* k,
                          const __half* v, const __half* q_obs, const float* scores_in, float* scores_out,
                          cudaStream_t st) {
  const Scratch& s = P.sc;
  const int nkb = (max_len + kKeyBlock - 1) / kKeyBlock;
  const dim3 grid(nkb, P.pv.hkv, n_req);
  cudaError_t e = cudaSuccess;
  const float* score_src;
  if (scores_in) {
    k_prompt_given<<<grid, 128, 0, st>>>(P.pv, scores_in, scores_out, s.tokinfo, s.bcnt, s.nkb_cap);
    e = cudaGetLastError();
    score_src = scores_in;
  } else {
    float* so = scores_out ? scores_out : s.score;
    e = launch_scoring_tc(P, k, q_obs, n_tok, n_req, so, st);
    score_src = so;
  }
  if (e != cudaSuccess) return e;
  if ((e = launch_prompt_plan(P, layer, n_req, st)) != cudaSuccess) return e;
  k_prompt_scatter<<<grid, 128, 0, st>>>(P.pv, s.tokinfo, s.bbase, s.rank2pos, s.nkb_cap);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const dim3 gpack((max_len + 32 * kPackGroups - 1) / (32 * kPackGroups), n_req * P.pv.hkv, 2);
  k_prompt_pack<<<gpack, 256, 0, st>>>(P.pv, k, v, score_src, s.rank2pos, s.unit_info, s.grant_ids, s.grant_cap);
  return cudaGetLastError();
}

}  // namespace dkv
