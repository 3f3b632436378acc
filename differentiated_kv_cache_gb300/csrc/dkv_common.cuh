// dkv_common.cuh — device-side definitions shared by the libdkv kernels.
//
// Everything here is GPU code written for sm_103a (GB300). The page format,
// free-list and table conventions are the ones stated in include/dkv.h; the
// method is DiffKV (SOSP'25): differentiated K/V precision, token-importance
// tiers and the parallel KV compaction memory manager.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dkv.h"

namespace dkv {

constexpr int kD = 128;            // head_dim
constexpr int kObs = 32;           // observation queries per prompt
constexpr int kMaxG = 8;           // query heads per KV head supported by the kernels
constexpr int kMaxCallReq = 1024;  // requests per call
constexpr int kTierPrune = 0, kTierLo = 1, kTierHi = 2, kTierMid = 3;   // mid: the optional third tier

// Geometry of one tier's unified page.
struct TierGeom {
  int t;          // tokens per page
  int kbytes;     // key row bytes (128 for 8-bit, 64 for 4-bit)
  int off[6];     // K codes, V codes, K meta, V meta, score, position
  uint32_t magic; // floor(2^32 / t) + 1: s / t == umulhi(s, magic) for s < 2^20

  __device__ __forceinline__ int div(int s) const { return (int)__umulhi((uint32_t)s, magic); }
};

// Device control block: free-list counters, sticky status, per-call flag.
struct Ctl {
  unsigned long long start;   // allocation counter
  unsigned long long end;     // reclaim counter
  int error;                  // sticky data-dependent error (0 = none); while set,
                              // every kernel of every call returns at once
  int error_info;
  int pad[2];
};

// Request slots of a call, passed by value to the per-step kernels.
struct SlotArgs {
  int n;
  int slots[kMaxCallReq];
};

// Per-call copy of the caller's host arrays (written by the set-up kernel).
struct CallArgs {
  int n_req;
  int pad;
  int slots[kMaxCallReq];
  int lens[kMaxCallReq];
  long long tok0[kMaxCallReq + 1];
};

// Least important tokens of one head: the argmin keys (order_key(importance)
// << 32 | position) of the hi tokens outside the recent window and of the lo
// tokens, their slots (-1: none), and the hi slot and importance of t_c (-1:
// not there). A partial covers part of a head's slots.
struct ScanPart {
  unsigned long long kh, kl;
  int sh, sl;
  int xc;
  float ic;
  unsigned long long km;      // mid tier (three-tier pools): argmin key and slot
  int sm, pad;
};

// One warp's share of a head's victim keys as the next generation step will
// see them, left by the score update of a decode-attention call: the argmin
// keys and slots of the hi tokens outside the next step's window, of the lo
// tokens and of the mid tokens among the warp's slots, and the hi slot and
// importance of t_c if the warp holds it (-1 otherwise). Every partial is
// stamped with the request's length N and update count after that call and
// with the number of partials the call left for the head; the head's first
// block also writes these stamps into a small array of their own (one 16-byte
// entry per head, read by every CTA of the next step's plan). A generation
// step reduces a head's partials while its stamps still match the request
// state, else it scans the head.
struct VictimPart {
  unsigned long long kh, kl, km;
  int sh, sl, sm, xc;
  float ic;
  int n_stamp, u_stamp, count;
};

// Device view of a pool, passed by value to every kernel.
struct PoolView {
  uint8_t* pages;
  int* list;
  int* table;        // [layer][slot][kvh][L]
  int* counts;       // [layer][slot][kvh][4]: hi tok, lo tok, hi pages, lo pages
  int* req;          // [layer][slot][4]: active, N0, N, updates
  Ctl* ctl;
  CallArgs* call;
  VictimPart* vparts;   // [layer][slot][kvh][max_vp]
  int4* vstamp;         // [layer][slot][kvh]: {N, update count, partials, 0} of the call that left them
  float2* alpha;        // [layer][kvh]: the head's (alpha_h, alpha_l)
  float* alpha_m;       // [layer][kvh]: the head's alpha_m (three-tier pools)
  int n_pages, page_bytes, n_layers, hkv, G, max_req, max_seq, L;
  int lo_enabled, window, slack, reclaim;
  // Three-tier pools: a row is the two-way table (L entries) followed by the
  // one-way mid table (Lm entries); counters are {hi tok, lo tok, hi pages,
  // lo pages, mid tok, mid pages, 0, 0}. Two-tier pools: Lm = 0, 4 counters.
  int mid_enabled, Lm, Lrow, cstride;
  int max_vp;           // victim-key partials per head (epilogue blocks x warps)
  TierGeom hi, lo, mid;

  __device__ __forceinline__ int* row(int layer, int slot, int kvh) const {
    return table + ((size_t)((size_t)layer * max_req + slot) * hkv + kvh) * Lrow;
  }
  __device__ __forceinline__ int* cnt(int layer, int slot, int kvh) const {
    return counts + ((size_t)((size_t)layer * max_req + slot) * hkv + kvh) * cstride;
  }
  // table entry of a tier's page k: hi from the left of the two-way part, lo
  // from its right, mid in the one-way part after it
  __device__ __forceinline__ int entry(int tier, int k) const {
    return tier == kTierHi ? k : (tier == kTierLo ? L - 1 - k : L + k);
  }
  __device__ __forceinline__ const TierGeom& geom(int tier) const {
    return tier == kTierHi ? hi : (tier == kTierLo ? lo : mid);
  }
  __device__ __forceinline__ int4* vst(int layer, int slot, int kvh) const {
    return vstamp + ((size_t)layer * max_req + slot) * hkv + kvh;
  }
  __device__ __forceinline__ VictimPart* vpart(int layer, int slot, int kvh) const {
    return vparts + (((size_t)layer * max_req + slot) * hkv + kvh) * max_vp;
  }
  __device__ __forceinline__ float2 thresholds(int layer, int kvh) const {
    return alpha[(size_t)layer * hkv + kvh];
  }
  __device__ __forceinline__ int* rq(int layer, int slot) const {
    return req + ((size_t)layer * max_req + slot) * 4;
  }
  __device__ __forceinline__ uint8_t* page(int id) const {
    return pages + (size_t)id * page_bytes;
  }
  // Sticky status set by an earlier kernel of the stream (visible at kernel
  // start). Read through L1: the first warp of an SM fetches the line and the
  // others hit, instead of every warp of a large grid queueing on the same
  // L2 line.
  __device__ __forceinline__ bool noop() const { return __ldca(&ctl->error) != 0; }
  // The same status read from L2, for a programmatic dependent after its
  // griddepcontrol.wait: an error its primary latched may postdate the line
  // an L1 read at the kernel's start fetched.
  __device__ __forceinline__ bool noop_after_wait() const { return *(volatile int*)&ctl->error != 0; }
};

// ---------------------------------------------------------------------------
// Importance count and three-way tier decision, fp32 correctly rounded.
// DiffKV, compaction policy: importance = mean attention received, compared
// with alpha_h/N and alpha_l/N; GQA heads combined with max.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int score_count(int j, int n0, int updates) {
  int c = (j < n0 ? min(n0 - j, kObs) : 0) + updates - (j >= n0 ? j - n0 : 0);
  return c < 1 ? 1 : c;
}

__device__ __forceinline__ int classify(float imp, float th_h, float th_l, int lo_enabled) {
  if (lo_enabled) {
    if (imp > th_h) return kTierHi;
    if (imp >= th_l) return kTierLo;
    return kTierPrune;
  }
  return imp >= th_l ? kTierHi : kTierPrune;
}

// Four-way decision of a three-tier pool (DiffKV, compaction policy:
// extensibility to more precision levels): hi above alpha_h/N, mid from
// alpha_m/N, lo from alpha_l/N, else pruned.
__device__ __forceinline__ int classify3(float imp, float th_h, float th_m, float th_l) {
  if (imp > th_h) return kTierHi;
  if (imp >= th_m) return kTierMid;
  if (imp >= th_l) return kTierLo;
  return kTierPrune;
}

// precision order of the tiers: prune < lo < mid < hi
__device__ __forceinline__ int tier_rank(int tier) {
  return tier == kTierHi ? 3 : (tier == kTierMid ? 2 : (tier == kTierLo ? 1 : 0));
}

// Total order on floats as unsigned keys (for argmin reductions).
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// ---------------------------------------------------------------------------
// Quantization codec (DiffKV, background: Q = round((X - z)/s), X^ = sQ + z),
// per token vector, every step an IEEE operation with explicit rounding so
// the codes are identical to any other correctly rounded implementation.
// ---------------------------------------------------------------------------
struct QParams {
  float inv;        // 1/s (unused when s == 0)
  float z;
  uint16_t sh, zh;  // fp16 bits of scale and zero
  bool zero_scale;
};

__device__ __forceinline__ QParams qparams(float mn, float mx, int bits) {
  QParams q;
  if (mn == 0.0f) mn = 0.0f;  // -0 taken as +0
  const float L = (float)((1 << bits) - 1);
  float s32 = __fdiv_rn(__fsub_rn(mx, mn), L);
  __half sh = __float2half_rn(s32), zh = __float2half_rn(mn);
  float s = __half2float(sh);
  q.z = __half2float(zh);
  q.sh = __half_as_ushort(sh);
  q.zh = __half_as_ushort(zh);
  q.zero_scale = (s == 0.0f);
  q.inv = q.zero_scale ? 0.0f : __frcp_rn(s);
  return q;
}

__device__ __forceinline__ uint32_t qcode(float x, const QParams& q, int bits) {
  if (q.zero_scale) return 0u;
  float t = __fmul_rn(__fsub_rn(x, q.z), q.inv);
  float r = rintf(t);
  r = fmaxf(r, 0.0f);
  r = fminf(r, (float)((1 << bits) - 1));
  return (uint32_t)r;
}

// Packed fp32 pairs (two IEEE fp32 operations per instruction, each correctly
// rounded like its scalar form).
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// clamp(rint_even(t), 0, 255) in one conversion (NaN gives 0); the 8-bit
// result is zero-extended into the 32-bit register
__device__ __forceinline__ uint32_t rint_sat_u8(float t) {
  uint32_t r;
  asm("cvt.rni.sat.u8.f32 %0, %1;\n" : "=r"(r) : "f"(t));
  return r;
}
// codes of the pair (x0, x1) under q, with the same arithmetic as qcode
__device__ __forceinline__ void qcode2(float x0, float x1, const QParams& q, int bits, uint32_t& c0, uint32_t& c1) {
  if (q.zero_scale) {
    c0 = c1 = 0u;
    return;
  }
  const uint64_t t = mul_f32x2(sub_f32x2(f32x2(x0, x1), f32x2(q.z, q.z)), f32x2(q.inv, q.inv));
  const uint32_t L = (1u << bits) - 1u;
  c0 = min(rint_sat_u8(__uint_as_float((uint32_t)t)), L);
  c1 = min(rint_sat_u8(__uint_as_float((uint32_t)(t >> 32))), L);
}

__device__ __forceinline__ float dequant(uint16_t sh, uint16_t zh, uint32_t code) {
  return __fmaf_rn(__half2float(__ushort_as_half(sh)), (float)code, __half2float(__ushort_as_half(zh)));
}

// bit offset of (feature f, slot-in-row e) inside value word f/4
__device__ __forceinline__ int vbit(int vbits, int f, int e) {
  int i = f & 3;
  return vbits == 4 ? 16 * e + 4 * i : 16 * (e & 1) + 4 * i + 2 * (e >> 1);
}

// ---------------------------------------------------------------------------
// PTX wrappers (legacy-MMA tensor path, async copies, warp matrix moves).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t* r, uint32_t smem_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte async global->shared copy; src_bytes = 0 zero-fills without reading.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
  uint32_t d;  // (a & mask) | orv
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(d) : "r"(a), "r"(mask), "r"(orv));
  return d;
}
__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b),
                      *reinterpret_cast<__half2*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
// (a, b) as the sum of two fp16 pairs: hi = fp16(x), lo = fp16(x - hi), about
// 22 significant bits together.
__device__ __forceinline__ void split_half2(float a, float b, uint32_t& hi, uint32_t& lo) {
  __half2 h = __floats2half2_rn(a, b);
  const float2 f = __half22float2(h);
  __half2 l = __floats2half2_rn(a - f.x, b - f.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}

// mbarrier + bulk asynchronous copy (global -> shared, completion counted in bytes)
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait that may suspend the thread for up to `ns` nanoseconds before
// reporting an incomplete phase (no busy spinning while copies are in flight)
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// Wait for a phase with a time bound (about one second); false on expiry.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_hint(bar, parity, 200000u)) {
    if (clock64() - t0 > 2000000000LL) return false;
  }
  return true;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }

// Programmatic dependent launch: a primary grid lets the next kernel on the
// stream launch early; that kernel waits for the primary's completion (and
// the visibility of its writes) before touching what the primary produced.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace dkv
