// decode_compact.cu — generation-phase compaction (DiffKV, compaction policy:
// generation phase and algorithm flow; memory management: generation
// workflow). One token per step per head:
//   1. the newest token enters the recent window, quantized hi;
//   2. the window's oldest token t_c is classified against alpha_h/N and
//      alpha_l/N (and alpha_m/N in a three-tier pool): it stays hi, is
//      re-quantized to lo (or mid), or is pruned;
//   3. if t_c was kept, the least important token t_v of its tier (hi: outside
//      the window) is considered for demotion (to the tier it classifies at)
//      or pruning.
// Removal from a tier fills the hole with the tier's last token. The per-head
// plan is made by k_decode_plan; pages are granted by k_decode_alloc
// (alloc.cu); k_decode_apply writes the token slots.
#include <algorithm>

#include "dkv_kernels.cuh"

namespace dkv {

constexpr int kPlanThreads = 256;

__device__ __forceinline__ float key_importance(unsigned long long key) {
  const uint32_t k = (uint32_t)(key >> 32);
  const uint32_t b = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(b);
}

// The scan of a head's slots is cut into CTAs of kScanSlots slots (hi slots,
// then lo slots); each CTA leaves its partial (least important hi token
// outside the window, least important lo token, the slot of t_c) and the last
// CTA of the head (per-head arrival counter, no waiting) reduces the partials
// and makes the plan.
constexpr int kScanSlots = kPlanThreads * 8;   // 2048: the pool sizes its scan partials with it

// What a head's plan needs besides its victim keys, loaded at the plan
// kernel's start with the request state (one round of loads for both): the
// length after the append, the tier counts and page counts before the step,
// and the head's thresholds.
struct HeadIn {
  int n, nh, nl, nm, php, plp, pmp;
  float2 al;
  float am;
};

template <bool MID>
__device__ __forceinline__ HeadIn load_head(const PoolView& pv, int layer, int slot, int kvh, int n) {
  const int* cn = pv.cnt(layer, slot, kvh);
  const int4 c4 = *reinterpret_cast<const int4*>(cn);   // counter rows start on 16-byte boundaries
  const int2 m2 = MID ? *reinterpret_cast<const int2*>(cn + 4) : make_int2(0, 0);
  return HeadIn{n, c4.x, c4.y, m2.x, c4.z, c4.w, m2.y, pv.thresholds(layer, kvh),
                MID ? pv.alpha_m[(size_t)layer * pv.hkv + kvh] : 0.0f};
}

// The plan of one head (one thread): bh / bl / bm the least important hi
// token outside the window, lo token and mid token (three-tier pools, MID),
// xc / ic the hi slot and importance of t_c; h the head's state.
template <bool MID>
__device__ void decide_plan(const PoolView& pv, const HeadIn& h, int unit, ArgMin bh, ArgMin bl, ArgMin bm,
                            int xc_in, float ic_in, DecodePlan* plans) {
  const int n = h.n;
  const int nh = h.nh, nl = h.nl, php = h.php, plp = h.plp;
  constexpr bool three = MID;
  const int nm = three ? h.nm : 0, pmp = three ? h.pmp : 0;
  const int pc = n - pv.window - 1;
  int s_xc = xc_in;
  float s_ic = ic_in;
  const float2 al = h.al;                        // the head's pair
  const float th_h = __fdiv_rn(al.x, (float)n), th_l = __fdiv_rn(al.y, (float)n);
  const float th_m = three ? __fdiv_rn(h.am, (float)n) : 0.0f;
  auto cls = [&](float imp) { return three ? classify3(imp, th_h, th_m, th_l) : classify(imp, th_h, th_l, pv.lo_enabled); };
  DecodePlan p;
  p.err = 0;
  p.n_moves = 0;
  int nh2 = nh + 1, nl2 = nl, nm2 = nm;       // (1) newest token appended at hi slot nh
  Move newmv{kTierHi, nh, kSrcNew, -1, kTierHi};
  if (pc >= 0) {
    const int xc = s_xc;
    if (xc < 0) {
      p.err = DKV_ERR_CHECK;
    } else {
      const int tc = cls(s_ic);
      if (tc == kTierHi) {
        // (3) hi victim: least important hi token outside the window (t_c
        // included); kept unless it classifies lower
        const int xv = bh.slot;
        const int cv = cls(key_importance(bh.key));
        if (cv != kTierHi) {
          newmv.dst_slot = xv;                // last (newest) token fills the hole
          nh2 = nh;
          if (cv == kTierLo) {
            p.mv[p.n_moves++] = Move{kTierLo, nl, kSrcDemote, xv, kTierHi};
            nl2 = nl + 1;
          } else if (cv == kTierMid) {
            p.mv[p.n_moves++] = Move{kTierMid, nm, kSrcDemote, xv, kTierHi};
            nm2 = nm + 1;
          }
        }
      } else if (tc == kTierLo || tc == kTierMid) {
        newmv.dst_slot = xc;                  // t_c leaves hi; the newest token fills it
        nh2 = nh;
        // t_c re-quantized and appended to its tier; that tier's victim over
        // its tokens and t_c
        const ArgMin bt = tc == kTierLo ? bl : bm;
        const int nt = tc == kTierLo ? nl : nm;
        const unsigned long long kc = ((unsigned long long)order_key(s_ic) << 32) | (uint32_t)pc;
        const bool tc_min = (bt.slot < 0) || (kc < bt.key);
        // t_c as the victim classifies at its own tier and stays
        const int cv = tc_min ? tc : cls(key_importance(bt.key));
        int nt2 = nt + 1;
        if (tier_rank(cv) < tier_rank(tc)) {
          // the victim leaves the tier; t_c fills its slot
          p.mv[p.n_moves++] = Move{tc, bt.slot, kSrcDemote, xc, kTierHi};
          nt2 = nt;
          if (cv == kTierLo) {                // a mid victim demoted to lo
            p.mv[p.n_moves++] = Move{kTierLo, nl, kSrcDemote, bt.slot, kTierMid};
            nl2 = nl + 1;
          }
        } else {
          p.mv[p.n_moves++] = Move{tc, nt, kSrcDemote, xc, kTierHi};
        }
        if (tc == kTierLo) nl2 = nt2; else nm2 = nt2;
      } else {
        newmv.dst_slot = xc;                  // t_c pruned
        nh2 = nh;
      }
    }
  }
  // the newest token's write goes last in the list: sources are read first anyway
  p.mv[p.n_moves++] = newmv;
  p.nh = nh2;
  p.nl = nl2;
  p.nm = nm2;
  const int need_h = (nh2 + pv.hi.t - 1) / pv.hi.t, need_l = (nl2 + pv.lo.t - 1) / pv.lo.t;
  p.new_hp = p.new_lp = p.free_hp = p.free_lp = p.new_mp = p.free_mp = 0;
  p.php = php;
  p.plp = plp;
  p.pmp = pmp;
  if (need_h > php) { p.new_hp = need_h - php; p.php = need_h; }
  else if (pv.reclaim && need_h < php) { p.free_hp = php - need_h; p.php = need_h; }
  if (need_l > plp) { p.new_lp = need_l - plp; p.plp = need_l; }
  else if (pv.reclaim && need_l < plp) { p.free_lp = plp - need_l; p.plp = need_l; }
  if (three) {
    const int need_m = (nm2 + pv.mid.t - 1) / pv.mid.t;
    if (need_m > pmp) { p.new_mp = need_m - pmp; p.pmp = need_m; }
    else if (pv.reclaim && need_m < pmp) { p.free_mp = pmp - need_m; p.pmp = need_m; }
  }
  if (p.err == 0 && (p.php + p.plp > pv.L || p.pmp > pv.Lm)) p.err = DKV_ERR_TABLE_FULL;
  plans[unit] = p;
}

// MID: a three-tier pool (the two-tier instance compiles the mid tier out)
template <bool MID>
__global__ void __launch_bounds__(kPlanThreads) k_decode_plan(PoolView pv, int layer, DecodePlan* plans,
                                                               ScanPart* parts, int* arrivals, int max_parts,
                                                               SlotArgs sa) {
  pdl_launch_dependents();        // k_decode_alloc may launch; it waits for this grid
  if (pv.noop()) return;
  __shared__ ArgMin s_tmp[(MID ? 3 : 2) * (kPlanThreads / 32)];
  __shared__ int s_xc, s_last;
  __shared__ float s_ic;
  const int c = blockIdx.x, kvh = blockIdx.y, i = blockIdx.z;
  const int slot = sa.slots[i];
  const int unit = i * pv.hkv + kvh;
  const int* rq = pv.rq(layer, slot);
  const int n0 = rq[1], n = rq[2] + 1, upd = rq[3];
  // the head's counts and thresholds, loaded in the same round as the
  // request state and the victim-key stamps below
  const HeadIn hin = load_head<MID>(pv, layer, slot, kvh, n);
  const int nh = hin.nh, nl = hin.nl, nm = hin.nm;
  // The victim-key partials the last decode-attention call's score update
  // left for this head, while the head is as that call left it (same length,
  // same update count): the first CTA's first warp reduces them (a partial
  // a lane), no scan. The condition is the same for every thread of the
  // head's CTAs.
  const VictimPart* vps = pv.vpart(layer, slot, kvh);
  const int4 vs4 = __ldcg(pv.vst(layer, slot, kvh));
  const int vcount = vs4.z;
  // The first warp of the head's first CTA loads up to 32 partials before it
  // knows whether they are valid, so that they arrive with the stamps (one
  // round of memory latency instead of two).
  ArgMin ch{~0ull, -1}, cl{~0ull, -1}, cm{~0ull, -1};
  int xc = -1;
  float ic = 0.0f;
  auto take = [&](const VictimPart* vp) {
    ch = amin(ch, ArgMin{__ldcg(&vp->kh), __ldcg(&vp->sh)});
    cl = amin(cl, ArgMin{__ldcg(&vp->kl), __ldcg(&vp->sl)});
    if (MID) cm = amin(cm, ArgMin{__ldcg(&vp->km), __ldcg(&vp->sm)});
    const int pxc = __ldcg(&vp->xc);
    const float pic = __ldcg(&vp->ic);
    if (pxc >= 0) {
      xc = pxc;
      ic = pic;
    }
  };
  if (c == 0 && threadIdx.x < 32 && threadIdx.x < pv.max_vp) take(vps + threadIdx.x);
  if (vs4.x == rq[2] && vs4.y == upd && vcount >= 1 && vcount <= pv.max_vp) {
    if (c != 0 || threadIdx.x >= 32) return;
    if (threadIdx.x >= vcount) {            // speculative loads past the call's partials
      ch = cl = cm = ArgMin{~0ull, -1};
      xc = -1;
    }
    for (int q = threadIdx.x + 32; q < vcount; q += 32) take(vps + q);
#pragma unroll
    for (int sft = 16; sft >= 1; sft >>= 1) {
      ch = shfl_amin(ch, sft);
      cl = shfl_amin(cl, sft);
      if (MID) cm = shfl_amin(cm, sft);
    }
    const unsigned has = __ballot_sync(0xffffffffu, xc >= 0);
    const int src = has ? __ffs(has) - 1 : 0;
    xc = __shfl_sync(0xffffffffu, xc, src);
    ic = __shfl_sync(0xffffffffu, ic, src);
    if (threadIdx.x == 0) decide_plan<MID>(pv, hin, unit, ch, cl, cm, xc, ic, plans);
    return;
  }
  const int nst = nh + nl + nm;             // slots: hi, then lo, then mid
  const int nparts = max(1, (nst + kScanSlots - 1) / kScanSlots);
  if (c >= nparts) return;
  const int* row = pv.row(layer, slot, kvh);
  const int pc = n - pv.window - 1;         // position of t_c
  const int wlim = n - pv.window;           // hi victims: position < wlim
  if (threadIdx.x == 0) { s_xc = -1; s_ic = 0.0f; }
  __syncthreads();
  ArgMin bh{~0ull, -1}, bl{~0ull, -1}, bm{~0ull, -1};
  // slots c*kScanSlots + k*kPlanThreads + tid: consecutive threads read
  // consecutive score / position entries of a page
  float sc[8];
  int pos[8], sl[8];
#pragma unroll
  for (int k = 0; k < 8; k++) {
    const int x = c * kScanSlots + k * kPlanThreads + threadIdx.x;
    sl[k] = -1;
    sc[k] = 0.0f;
    pos[k] = 0;
    if (x >= nst) continue;
    const int tier = x < nh ? kTierHi : (!MID || x < nh + nl ? kTierLo : kTierMid);
    const int s = x < nh ? x : (!MID || x < nh + nl ? x - nh : x - nh - nl);
    const TierGeom& tg = pv.geom(tier);
    const int d = tg.div(s);
    const uint8_t* pg = pv.page(__ldg(row + pv.entry(tier, d)));
    sc[k] = *reinterpret_cast<const float*>(pg + tg.off[4] + 4 * (s - d * tg.t));
    pos[k] = *reinterpret_cast<const int*>(pg + tg.off[5] + 4 * (s - d * tg.t));
    sl[k] = x;
  }
#pragma unroll
  for (int k = 0; k < 8; k++) {
    if (sl[k] < 0) continue;
    const float imp = __fdiv_rn(sc[k], (float)score_count(pos[k], n0, upd));
    const unsigned long long key = ((unsigned long long)order_key(imp) << 32) | (uint32_t)pos[k];
    if (sl[k] < nh) {
      if (pos[k] == pc) { s_xc = sl[k]; s_ic = imp; }
      if (pos[k] < wlim) bh = amin(bh, ArgMin{key, sl[k]});
    } else if (!MID || sl[k] < nh + nl) {
      bl = amin(bl, ArgMin{key, sl[k] - nh});
    } else {
      bm = amin(bm, ArgMin{key, sl[k] - nh - nl});
    }
  }
  if (MID) block_amin3(bh, bl, bm, s_tmp);
  else block_amin2(bh, bl, s_tmp);
  if (threadIdx.x == 0) {
    ScanPart& part = parts[(size_t)unit * max_parts + c];
    part.kh = bh.key; part.sh = bh.slot;
    part.kl = bl.key; part.sl = bl.slot;
    part.km = bm.key; part.sm = bm.slot;
    part.xc = s_xc; part.ic = s_ic;
    __threadfence();
    s_last = atomicAdd(arrivals + unit, 1) == nparts - 1;
  }
  __syncthreads();
  if (!s_last || threadIdx.x != 0) return;
  __threadfence();
  arrivals[unit] = 0;                       // ready for the next step
  ArgMin rh{~0ull, -1}, rl{~0ull, -1}, rm{~0ull, -1};
  int rx = -1;
  float ri = 0.0f;
  for (int q = 0; q < nparts; q++) {
    const ScanPart& part = parts[(size_t)unit * max_parts + q];
    const ArgMin ph{__ldcg(&part.kh), __ldcg(&part.sh)}, pl{__ldcg(&part.kl), __ldcg(&part.sl)};
    rh = amin(rh, ph);
    rl = amin(rl, pl);
    if (MID) rm = amin(rm, ArgMin{__ldcg(&part.km), __ldcg(&part.sm)});
    const int pxc = __ldcg(&part.xc);
    const float pic = __ldcg(&part.ic);
    if (pxc >= 0) { rx = pxc; ri = pic; }
  }
  decide_plan<MID>(pv, hin, unit, rh, rl, rm, rx, ri, plans);
}

// Token record staged in shared memory between the read and write phases.
struct TokStage {
  uint8_t kc[kD], vc[kD];
  uint32_t kmeta, vmeta;
  float score;
  int pos;
};

// Warp-wide min / max of one value per lane.
__device__ __forceinline__ void warp_minmax(float& mn, float& mx) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, s));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
  }
}

// Quantize 4 features per lane (features 4*lane..4*lane+3) into the stage.
__device__ __forceinline__ void warp_quantize(const float* x, int bits, uint8_t* codes, uint32_t* meta) {
  const int lane = threadIdx.x & 31;
  float mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
  float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  warp_minmax(mn, mx);
  const QParams q = qparams(mn, mx, bits);
#pragma unroll
  for (int e = 0; e < 4; e++) codes[4 * lane + e] = (uint8_t)qcode(x[e], q, bits);
  if (lane == 0) *meta = (uint32_t)q.sh | ((uint32_t)q.zh << 16);
}

template <bool MID>
__global__ void __launch_bounds__(64) k_decode_apply(PoolView pv, int layer, const DecodePlan* __restrict__ plans,
                                                      const __half* __restrict__ knew,
                                                      const __half* __restrict__ vnew, SlotArgs sa) {
  pdl_launch_dependents();        // a decode-attention call may follow: it waits for this grid
  if (pv.noop()) return;
  __shared__ TokStage st[3];      // [0], [1]: demoted sources of moves 0, 1; [2]: the new token
  const int kvh = blockIdx.x, i = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The new token's hi codes do not depend on the plan: warp 1 quantizes
  // them (from the caller's buffers) while the plan and allocation finish.
  if (warp == 1) {
    TokStage& s = st[2];
    const __half* kp = knew + ((size_t)i * pv.hkv + kvh) * kD + 4 * lane;
    const __half* vp = vnew + ((size_t)i * pv.hkv + kvh) * kD + 4 * lane;
    float kx[4], vx[4];
#pragma unroll
    for (int e = 0; e < 4; e++) { kx[e] = __half2float(kp[e]); vx[e] = __half2float(vp[e]); }
    warp_quantize(kx, 8, s.kc, &s.kmeta);
    warp_quantize(vx, 4, s.vc, &s.vmeta);
  }
  pdl_wait();                     // the plans and pages of k_decode_alloc
  if (pv.noop_after_wait()) return;
  const int slot = sa.slots[i];
  const int unit = i * pv.hkv + kvh;
  const DecodePlan& p = plans[unit];
  const int* row = pv.row(layer, slot, kvh);
  const int n = pv.rq(layer, slot)[2];       // already advanced by k_decode_alloc
  if (threadIdx.x == 0) { st[2].score = 0.0f; st[2].pos = n - 1; }
  // read phase: warp m stages the source of move m when it is a demotion
  // (the new token is always the last move, so m < 2)
  if (warp < p.n_moves && p.mv[warp].src != kSrcNew) {
    const Move mv = p.mv[warp];
    TokStage& s = st[warp];
    float kx[4], vx[4];
    {
      // demote: dequantize the source slot's codes (hi K8V4 or mid K8V2),
      // quantize again at the destination's precision (mid K8V2, lo K4V2)
      // a two-tier pool demotes hi -> lo only
      const int src_tier = MID ? mv.src_tier : kTierHi, dst_tier = MID ? mv.dst_tier : kTierLo;
      const TierGeom& sg = MID ? pv.geom(src_tier) : pv.hi;
      const int svb = src_tier == kTierHi ? 4 : 2, sgsz = 8 / svb;
      const int d = sg.div(mv.src_slot);
      const uint8_t* pg = pv.page(row[MID ? pv.entry(src_tier, d) : d]);
      const int ip = mv.src_slot - d * sg.t;
      const uint32_t km = *reinterpret_cast<const uint32_t*>(pg + sg.off[2] + 4 * ip);
      const uint32_t vm = *reinterpret_cast<const uint32_t*>(pg + sg.off[3] + 4 * ip);
      const uint32_t kw = *reinterpret_cast<const uint32_t*>(pg + sg.off[0] + ip * sg.kbytes + 4 * lane);
      const uint32_t vw = *reinterpret_cast<const uint32_t*>(pg + sg.off[1] + (ip / sgsz) * 128 + 4 * lane);
#pragma unroll
      for (int e = 0; e < 4; e++) {
        kx[e] = dequant((uint16_t)km, (uint16_t)(km >> 16), (kw >> (8 * e)) & 255u);
        vx[e] = dequant((uint16_t)vm, (uint16_t)(vm >> 16),
                        (vw >> vbit(svb, 4 * lane + e, ip % sgsz)) & ((1u << svb) - 1u));
      }
      warp_quantize(kx, dst_tier == kTierLo ? 4 : 8, s.kc, &s.kmeta);
      warp_quantize(vx, 2, s.vc, &s.vmeta);
      if (lane == 0) {
        s.score = *reinterpret_cast<const float*>(pg + sg.off[4] + 4 * ip);
        s.pos = *reinterpret_cast<const int*>(pg + sg.off[5] + 4 * ip);
      }
    }
  }
  __syncthreads();
  if (warp != 0) return;
  // write phase: one warp, moves in order (value words shared between slots)
  for (int m = 0; m < p.n_moves; m++) {
    const Move mv = p.mv[m];
    const TokStage& s = st[mv.src == kSrcNew ? 2 : m];
    const int tier = mv.dst_tier;
    const TierGeom& tg = MID ? pv.geom(tier) : (tier == kTierHi ? pv.hi : pv.lo);
    const int d = tg.div(mv.dst_slot);
    uint8_t* pg = pv.page(row[MID ? pv.entry(tier, d) : (tier == kTierHi ? d : pv.L - 1 - d)]);
    const int ip = mv.dst_slot - d * tg.t;
    const uint8_t* kc = s.kc + 4 * lane;
    if (tier != kTierLo) {                    // 8-bit keys (hi, mid)
      *reinterpret_cast<uint32_t*>(pg + tg.off[0] + ip * 128 + 4 * lane) =
          kc[0] | (kc[1] << 8) | (kc[2] << 16) | ((uint32_t)kc[3] << 24);
    } else {
      *reinterpret_cast<uint16_t*>(pg + tg.off[0] + ip * 64 + 2 * lane) =
          (uint16_t)(kc[0] | (kc[1] << 4) | (kc[2] << 8) | (kc[3] << 12));
    }
    const int vbits = tier == kTierHi ? 4 : 2, gsz = tier == kTierHi ? 2 : 4;
    uint32_t* vw = reinterpret_cast<uint32_t*>(pg + tg.off[1] + (ip / gsz) * 128) + lane;
    uint32_t w = *vw;
    const uint32_t lmask = (1u << vbits) - 1u;
#pragma unroll
    for (int e = 0; e < 4; e++) {
      const int b = vbit(vbits, 4 * lane + e, ip % gsz);
      w = (w & ~(lmask << b)) | ((uint32_t)s.vc[4 * lane + e] << b);
    }
    *vw = w;
    if (lane == 0) {
      *reinterpret_cast<uint32_t*>(pg + tg.off[2] + 4 * ip) = s.kmeta;
      *reinterpret_cast<uint32_t*>(pg + tg.off[3] + 4 * ip) = s.vmeta;
      *reinterpret_cast<float*>(pg + tg.off[4] + 4 * ip) = s.score;
      *reinterpret_cast<int*>(pg + tg.off[5] + 4 * ip) = s.pos;
    }
    __syncwarp();
  }
}

cudaError_t launch_decode_alloc(Pool& P, int layer, const SlotArgs& sa, cudaStream_t st);

cudaError_t launch_decode(Pool& P, int layer, const SlotArgs& sa, const __half* k, const __half* v,
                          cudaStream_t st) {
  const dim3 grid(P.pv.hkv, sa.n);
  int max_n = 1;
  for (int i = 0; i < sa.n; i++) max_n = std::max(max_n, P.h_n[(size_t)layer * P.cfg.max_requests + sa.slots[i]]);
  const int scan_ctas = (max_n + 1 + kScanSlots - 1) / kScanSlots;   // stored tokens of all tiers <= N + 1
  if (scan_ctas > P.sc.max_scan) return cudaErrorInvalidConfiguration;
  const dim3 gscan(scan_ctas, P.pv.hkv, sa.n);
  if (P.pv.mid_enabled)
    k_decode_plan<true><<<gscan, kPlanThreads, 0, st>>>(P.pv, layer, P.sc.dplan, P.sc.dscan, P.sc.darrive,
                                                        P.sc.max_scan, sa);
  else
    k_decode_plan<false><<<gscan, kPlanThreads, 0, st>>>(P.pv, layer, P.sc.dplan, P.sc.dscan, P.sc.darrive,
                                                         P.sc.max_scan, sa);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if ((e = launch_decode_alloc(P, layer, sa, st)) != cudaSuccess) return e;
  // a programmatic dependent of k_decode_alloc
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = dim3(64);
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (P.pv.mid_enabled)
    e = cudaLaunchKernelEx(&lc, k_decode_apply<true>, P.pv, layer, (const DecodePlan*)P.sc.dplan, k, v, sa);
  else
    e = cudaLaunchKernelEx(&lc, k_decode_apply<false>, P.pv, layer, (const DecodePlan*)P.sc.dplan, k, v, sa);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dkv
