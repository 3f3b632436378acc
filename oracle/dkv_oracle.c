/*
 * dkv_oracle.c — plain, slow CPU oracle of differentiated KV compaction.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline of the benchmark may load this library. It shares no code, header,
 * table or constant generator with the CUDA library; it is written directly
 * from "DiffKV: Differentiated Memory Management for Large Language Models
 * with Parallel KV Compaction" (SOSP'25) and from the page format stated in
 * the library's public header (a data format both sides must agree on).
 *
 * Precision: scores and attention in fp64; the quantization codec and the
 * tier comparisons in fp32 with every operation correctly rounded and no
 * contraction (compile with -ffp-contract=off), because those decide integers
 * that must match bit for bit.
 *
 * Section names cited below refer to the DiffKV page:
 *   Background (quantization; attention equation), Compaction policy
 *   (prompt phase; generation phase; algorithm flow), Memory management
 *   (parallel KV compaction; unified pages; circular free page list;
 *   bidirectional page table; prompt workflow, Figure 6; generation workflow).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG -1
#define ORC_ERR_STATE -3
#define ORC_ERR_NO_PAGES -4
#define ORC_ERR_TABLE_FULL -5
#define ORC_ERR_CHECK -7

#define D 128
#define OBS 32
#define TIER_PRUNE 0
#define TIER_LO 1
#define TIER_HI 2
#define TIER_MID 3   /* the optional third precision level, between hi and lo */

/* ------------------------------------------------------------------ */
/* IEEE binary16 <-> binary32, written from the IEEE 754 definition.   */
/* ------------------------------------------------------------------ */
float orc_half_to_float(uint16_t h) {
  int sign = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0) v = ldexp((double)m, -24);                 /* subnormal m * 2^-24 */
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(m + 1024), e - 25);            /* (1 + m/1024) 2^(e-15) */
  return (float)(sign ? -v : v);
}

uint16_t orc_float_to_half(float f) {
  /* round to nearest, ties to even (nearbyint in the default rounding mode) */
  uint16_t sign = signbit(f) ? 0x8000 : 0;
  if (isnan(f)) return sign | 0x7e00;
  double a = fabs((double)f);
  if (a >= 65520.0) return sign | 0x7c00;                /* past max + half ulp */
  if (a < ldexp(1.0, -14)) {                             /* subnormal range     */
    double m = nearbyint(a * ldexp(1.0, 24));            /* units of 2^-24      */
    return sign | (uint16_t)m;                           /* 1024 -> min normal  */
  }
  int ex;
  frexp(a, &ex);                                         /* a in [2^(ex-1), 2^ex) */
  double m = nearbyint(ldexp(a, 11 - ex));               /* in [1024, 2048]     */
  int biased = ex - 1 + 15;
  if (m == 2048.0) { m = 1024.0; biased += 1; }
  if (biased >= 31) return sign | 0x7c00;
  return sign | (uint16_t)(biased << 10) | (uint16_t)((int)m - 1024);
}

/* ------------------------------------------------------------------ */
/* Quantization codec — Background, quantization: Q = round((X-z)/s),  */
/* X^ = s Q + z, per key / value vector with its own scale and zero.   */
/* ------------------------------------------------------------------ */
void orc_quantize(const float* x, int n, int bits, uint8_t* code, uint16_t* scale_h,
                  uint16_t* zero_h) {
  const int L = (1 << bits) - 1;
  float mn = x[0], mx = x[0];
  for (int i = 1; i < n; i++) {
    if (x[i] < mn) mn = x[i];
    if (x[i] > mx) mx = x[i];
  }
  if (mn == 0.0f) mn = 0.0f;                             /* -0 is taken as +0 */
  float range = mx - mn;
  float s32 = range / (float)L;
  uint16_t sh = orc_float_to_half(s32), zh = orc_float_to_half(mn);
  float s = orc_half_to_float(sh), z = orc_half_to_float(zh);
  if (s == 0.0f) {
    for (int i = 0; i < n; i++) code[i] = 0;
  } else {
    float inv = 1.0f / s;
    for (int i = 0; i < n; i++) {
      float t = (x[i] - z) * inv;
      float r = rintf(t);
      if (r < 0.0f) r = 0.0f;
      if (r > (float)L) r = (float)L;
      code[i] = (uint8_t)r;
    }
  }
  *scale_h = sh;
  *zero_h = zh;
}

float orc_dequant(uint16_t scale_h, uint16_t zero_h, int code) {
  return fmaf(orc_half_to_float(scale_h), (float)code, orc_half_to_float(zero_h));
}

/* ------------------------------------------------------------------ */
/* Pool state — Memory management: unified pages, circular free page   */
/* list, bidirectional page table.                                     */
/* ------------------------------------------------------------------ */
typedef struct {
  int32_t n_layers, n_kv_heads, group_size, page_bytes, n_pages, max_requests, max_seq_len;
  int32_t t_hi, t_lo;          /* 0 = derive from page_bytes */
  int32_t lo_enabled;
  float alpha_h, alpha_l;
  int32_t window, grant_slack, reclaim_in_decode;
  int32_t mid_enabled;         /* 1: a third level K8V2 between hi and lo */
  float alpha_m;               /* its threshold alpha_m / N */
  int32_t t_mid;               /* 0 = derive from page_bytes */
} orc_config;

typedef struct {
  int t;                       /* tokens per page */
  int kbits, vbits, g;         /* g = tokens sharing one value byte */
  int off[6];                  /* K codes, V codes, K meta, V meta, score, position */
  int used;
} tier_geom;

typedef struct {
  orc_config c;
  tier_geom tg[4];             /* indexed by TIER_LO / TIER_HI / TIER_MID */
  int table_len;               /* entries of the two-way part of a row (hi | lo) */
  int mid_len;                 /* entries of the one-way part (mid pages), 0 without mid */
  int row_len;                 /* table_len + mid_len */
  int cstride;                 /* ints of per-head counters: 4, or 8 with mid */
  uint8_t* pages;
  int32_t* list;
  int64_t ptr[2];              /* start, end */
  int32_t* table;              /* [layer][slot][kvh][row_len] */
  int32_t* counts;             /* [layer][slot][kvh][cstride] hi tok, lo tok, hi pages, lo pages
                                  (then mid tok, mid pages, 0, 0 with mid) */
  int32_t* req;                /* [layer][slot][4] active, N0, N, updates */
  float* alpha;                /* [layer][kvh][2] alpha_h, alpha_l of each head */
  float* alpha_mid;            /* [layer][kvh] alpha_m of each head */
} orc_pool;

static int round16(int x) { return (x + 15) & ~15; }

static void layout(tier_geom* g, int t) {
  g->t = t;
  int sz[6] = {t * D * g->kbits / 8, (t / g->g) * 128, 4 * t, 4 * t, 4 * t, 4 * t};
  int o = 0;
  for (int i = 0; i < 6; i++) {
    g->off[i] = o;
    o = round16(o + sz[i]);
  }
  g->used = g->off[5] + sz[5];
}

static int fit_tokens(tier_geom* g, int page_bytes) {
  int best = 0;
  for (int t = g->g; t <= page_bytes; t += g->g) {
    layout(g, t);
    if (g->used <= page_bytes) best = t; else break;
  }
  return best;
}

static int32_t* trow(orc_pool* p, int layer, int slot, int kvh) {
  return p->table + (((int64_t)layer * p->c.max_requests + slot) * p->c.n_kv_heads + kvh) * p->row_len;
}
static int32_t* hcnt(orc_pool* p, int layer, int slot, int kvh) {
  return p->counts + (((int64_t)layer * p->c.max_requests + slot) * p->c.n_kv_heads + kvh) * p->cstride;
}
static int32_t* rstate(orc_pool* p, int layer, int slot) {
  return p->req + ((int64_t)layer * p->c.max_requests + slot) * 4;
}
static uint8_t* page_ptr(orc_pool* p, int page) { return p->pages + (int64_t)page * p->c.page_bytes; }

orc_pool* orc_pool_new(const orc_config* c) {
  orc_pool* p = (orc_pool*)calloc(1, sizeof(orc_pool));
  p->c = *c;
  p->tg[TIER_HI].kbits = 8; p->tg[TIER_HI].vbits = 4; p->tg[TIER_HI].g = 2;
  p->tg[TIER_LO].kbits = 4; p->tg[TIER_LO].vbits = 2; p->tg[TIER_LO].g = 4;
  p->tg[TIER_MID].kbits = 8; p->tg[TIER_MID].vbits = 2; p->tg[TIER_MID].g = 4;
  int th = c->t_hi ? c->t_hi : fit_tokens(&p->tg[TIER_HI], c->page_bytes);
  int tl = c->t_lo ? c->t_lo : fit_tokens(&p->tg[TIER_LO], c->page_bytes);
  int tm = c->t_mid ? c->t_mid : fit_tokens(&p->tg[TIER_MID], c->page_bytes);
  layout(&p->tg[TIER_HI], th);
  layout(&p->tg[TIER_LO], tl);
  layout(&p->tg[TIER_MID], tm);
  /* Bidirectional page table entry length: max sequence length over tokens per
   * hi page, plus one page for a hi/lo split whose two partial pages exceed it. */
  p->table_len = (c->max_seq_len + th - 1) / th + 1;
  /* With a third level the row composes the two-way table with a one-way
   * table of mid pages (Memory management, generation workflow: further
   * precision levels by combining one-way or two-way page tables). */
  p->mid_len = c->mid_enabled ? (c->max_seq_len + tm - 1) / tm + 1 : 0;
  p->row_len = p->table_len + p->mid_len;
  p->cstride = c->mid_enabled ? 8 : 4;
  p->pages = (uint8_t*)calloc((size_t)c->n_pages, (size_t)c->page_bytes);
  p->list = (int32_t*)malloc(sizeof(int32_t) * (size_t)c->n_pages);
  for (int i = 0; i < c->n_pages; i++) p->list[i] = i;
  p->ptr[0] = 0;
  p->ptr[1] = c->n_pages;
  size_t heads = (size_t)c->n_layers * c->max_requests * c->n_kv_heads;
  p->table = (int32_t*)malloc(sizeof(int32_t) * heads * p->row_len);
  for (size_t i = 0; i < heads * p->row_len; i++) p->table[i] = -1;
  p->counts = (int32_t*)calloc(heads * p->cstride, sizeof(int32_t));
  p->req = (int32_t*)calloc((size_t)c->n_layers * c->max_requests * 4, sizeof(int32_t));
  /* every head starts with the configuration's thresholds */
  p->alpha = (float*)malloc(sizeof(float) * 2 * (size_t)c->n_layers * c->n_kv_heads);
  for (int x = 0; x < c->n_layers * c->n_kv_heads; x++) {
    p->alpha[2 * x] = c->alpha_h;
    p->alpha[2 * x + 1] = c->alpha_l;
  }
  p->alpha_mid = (float*)malloc(sizeof(float) * (size_t)c->n_layers * c->n_kv_heads);
  for (int x = 0; x < c->n_layers * c->n_kv_heads; x++) p->alpha_mid[x] = c->alpha_m;
  return p;
}

/* Compaction policy, extensibility: thresholds set for each head on its own
 * (here per layer and KV head). Later steps of `layer` compare head h's
 * tokens with ah[h]/N and al[h]/N. */
int orc_set_thresholds(orc_pool* p, int layer, const float* ah, const float* al) {
  if (layer < 0 || layer >= p->c.n_layers || !ah || !al) return ORC_ERR_ARG;
  for (int h = 0; h < p->c.n_kv_heads; h++) {
    if (isnan(ah[h]) || isnan(al[h])) return ORC_ERR_ARG;
  }
  for (int h = 0; h < p->c.n_kv_heads; h++) {
    p->alpha[2 * ((size_t)layer * p->c.n_kv_heads + h)] = ah[h];
    p->alpha[2 * ((size_t)layer * p->c.n_kv_heads + h) + 1] = al[h];
  }
  return ORC_OK;
}

float* orc_thresholds(orc_pool* p) { return p->alpha; }

/* The mid level's threshold of each head of `layer` (am[h]/N). */
int orc_set_mid_thresholds(orc_pool* p, int layer, const float* am) {
  if (layer < 0 || layer >= p->c.n_layers || !am || !p->c.mid_enabled) return ORC_ERR_ARG;
  for (int h = 0; h < p->c.n_kv_heads; h++)
    if (isnan(am[h])) return ORC_ERR_ARG;
  for (int h = 0; h < p->c.n_kv_heads; h++) p->alpha_mid[(size_t)layer * p->c.n_kv_heads + h] = am[h];
  return ORC_OK;
}

float* orc_mid_thresholds(orc_pool* p) { return p->alpha_mid; }

void orc_pool_free(orc_pool* p) {
  if (!p) return;
  free(p->pages); free(p->list); free(p->table); free(p->counts); free(p->req); free(p->alpha);
  free(p->alpha_mid);
  free(p);
}

/* geometry: t_hi, t_lo, table_len, hi off[6], lo off[6], hi used, lo used,
 * t_mid, mid_len, mid off[6], mid used, row_len, cstride */
void orc_geometry(const orc_pool* p, int32_t* out) {
  out[0] = p->tg[TIER_HI].t;
  out[1] = p->tg[TIER_LO].t;
  out[2] = p->table_len;
  for (int i = 0; i < 6; i++) out[3 + i] = p->tg[TIER_HI].off[i];
  for (int i = 0; i < 6; i++) out[9 + i] = p->tg[TIER_LO].off[i];
  out[15] = p->tg[TIER_HI].used;
  out[16] = p->tg[TIER_LO].used;
  out[17] = p->tg[TIER_MID].t;
  out[18] = p->mid_len;
  for (int i = 0; i < 6; i++) out[19 + i] = p->tg[TIER_MID].off[i];
  out[25] = p->tg[TIER_MID].used;
  out[26] = p->row_len;
  out[27] = p->cstride;
}

uint8_t* orc_pages(orc_pool* p) { return p->pages; }
int32_t* orc_list(orc_pool* p) { return p->list; }
int64_t* orc_pointers(orc_pool* p) { return p->ptr; }
int32_t* orc_table(orc_pool* p) { return p->table; }
int32_t* orc_head_counts(orc_pool* p) { return p->counts; }
int32_t* orc_req_state(orc_pool* p) { return p->req; }

/* ------------------------------------------------------------------ */
/* One token record and its placement in a unified page.               */
/* ------------------------------------------------------------------ */
typedef struct {
  uint8_t kc[D], vc[D];        /* codes at the record's tier */
  uint16_t ks, kz, vs, vz;     /* fp16 bits */
  float score;
  int32_t pos;
} token_rec;

static uint32_t rd32(const uint8_t* b) {
  return (uint32_t)b[0] | ((uint32_t)b[1] << 8) | ((uint32_t)b[2] << 16) | ((uint32_t)b[3] << 24);
}
static void wr32(uint8_t* b, uint32_t v) {
  b[0] = (uint8_t)v; b[1] = (uint8_t)(v >> 8); b[2] = (uint8_t)(v >> 16); b[3] = (uint8_t)(v >> 24);
}
static void wr16(uint8_t* b, uint16_t v) { b[0] = (uint8_t)v; b[1] = (uint8_t)(v >> 8); }
static uint16_t rd16(const uint8_t* b) { return (uint16_t)(b[0] | (b[1] << 8)); }

/* bit offset of (feature f, slot-in-row e) inside value word f/4 */
static int vbit(int vbits, int f, int e) {
  int i = f & 3;
  if (vbits == 4) return 16 * e + 4 * i;
  return 16 * (e & 1) + 4 * i + 2 * (e >> 1);
}

static void put_token(uint8_t* page, const tier_geom* g, int slot, const token_rec* r) {
  /* key row: 8-bit one byte per feature; 4-bit two features per byte, low nibble first */
  uint8_t* krow = page + g->off[0] + slot * (D * g->kbits / 8);
  if (g->kbits == 8) {
    for (int f = 0; f < D; f++) krow[f] = r->kc[f];
  } else {
    for (int b = 0; b < D / 2; b++) krow[b] = (uint8_t)((r->kc[2 * b] & 15) | ((r->kc[2 * b + 1] & 15) << 4));
  }
  /* value row shared by g consecutive slots */
  uint8_t* vrow = page + g->off[1] + (slot / g->g) * 128;
  int e = slot % g->g;
  uint32_t lmask = (1u << g->vbits) - 1;
  for (int w = 0; w < 32; w++) {
    uint32_t word = rd32(vrow + 4 * w);
    for (int i = 0; i < 4; i++) {
      int f = 4 * w + i, bit = vbit(g->vbits, f, e);
      word &= ~(lmask << bit);
      word |= ((uint32_t)r->vc[f] & lmask) << bit;
    }
    wr32(vrow + 4 * w, word);
  }
  wr16(page + g->off[2] + 4 * slot, r->ks);
  wr16(page + g->off[2] + 4 * slot + 2, r->kz);
  wr16(page + g->off[3] + 4 * slot, r->vs);
  wr16(page + g->off[3] + 4 * slot + 2, r->vz);
  memcpy(page + g->off[4] + 4 * slot, &r->score, 4);
  memcpy(page + g->off[5] + 4 * slot, &r->pos, 4);
}

static void get_token(const uint8_t* page, const tier_geom* g, int slot, token_rec* r) {
  const uint8_t* krow = page + g->off[0] + slot * (D * g->kbits / 8);
  if (g->kbits == 8) {
    for (int f = 0; f < D; f++) r->kc[f] = krow[f];
  } else {
    for (int b = 0; b < D / 2; b++) { r->kc[2 * b] = krow[b] & 15; r->kc[2 * b + 1] = krow[b] >> 4; }
  }
  const uint8_t* vrow = page + g->off[1] + (slot / g->g) * 128;
  int e = slot % g->g;
  uint32_t lmask = (1u << g->vbits) - 1;
  for (int f = 0; f < D; f++) r->vc[f] = (uint8_t)((rd32(vrow + 4 * (f / 4)) >> vbit(g->vbits, f, e)) & lmask);
  r->ks = rd16(page + g->off[2] + 4 * slot);
  r->kz = rd16(page + g->off[2] + 4 * slot + 2);
  r->vs = rd16(page + g->off[3] + 4 * slot);
  r->vz = rd16(page + g->off[3] + 4 * slot + 2);
  memcpy(&r->score, page + g->off[4] + 4 * slot, 4);
  memcpy(&r->pos, page + g->off[5] + 4 * slot, 4);
}

/* quantize fp32 K and V vectors of one token at a tier */
static void make_token(const float* k, const float* v, const tier_geom* g, float score, int pos,
                       token_rec* r) {
  orc_quantize(k, D, g->kbits, r->kc, &r->ks, &r->kz);
  orc_quantize(v, D, g->vbits, r->vc, &r->vs, &r->vz);
  r->score = score;
  r->pos = pos;
}

static void half_vec(const uint16_t* h, float* out) {
  for (int i = 0; i < D; i++) out[i] = orc_half_to_float(h[i]);
}

/* Re-quantization of a stored token to another level (hi -> lo, hi -> mid,
 * mid -> lo): dequantize its codes, quantize the values again */
static void requant(const token_rec* src, const tier_geom* dst, token_rec* out) {
  float k[D], v[D];
  for (int f = 0; f < D; f++) {
    k[f] = orc_dequant(src->ks, src->kz, src->kc[f]);
    v[f] = orc_dequant(src->vs, src->vz, src->vc[f]);
  }
  make_token(k, v, dst, src->score, src->pos, out);
}

/* page holding slot s of a tier (through the head's table row: hi pages from
 * the left of the two-way part, lo pages from its right, mid pages in the
 * one-way part after it) and the slot's index inside that page */
static uint8_t* slot_loc(orc_pool* p, const int32_t* row, int tier, int s, int* in_page) {
  const int t = p->tg[tier].t;
  *in_page = s % t;
  int e = tier == TIER_HI ? s / t : tier == TIER_LO ? p->table_len - 1 - s / t : p->table_len + s / t;
  return page_ptr(p, row[e]);
}

/* ------------------------------------------------------------------ */
/* Importance and tiers — Compaction policy.                           */
/* ------------------------------------------------------------------ */

/* Number of attention scores summed into a token's score: the observation
 * queries at or after it (prompt), plus one per score update since it was
 * stored (generation; a token generated at decode step j-N0 has seen
 * updates-(j-N0) queries). Never below 1. */
static int score_count(int j, int n0, int updates) {
  int c = (j < n0 ? (n0 - j < OBS ? n0 - j : OBS) : 0) + updates - (j >= n0 ? j - n0 : 0);
  return c < 1 ? 1 : c;
}

static float importance(float score, int count) { return score / (float)count; }

/* three-way split against alpha_h/N and alpha_l/N (the head's thresholds);
 * with the lo tier disabled a token that would be lo is kept at hi precision;
 * with the mid level a token at or above alpha_m/N that is not hi is mid.
 * alpha: the head's {alpha_h, alpha_l}; am: its alpha_m. */
static int classify(const orc_config* c, const float* alpha, float am, float imp, int n) {
  float th_h = alpha[0] / (float)n, th_l = alpha[1] / (float)n;
  if (c->lo_enabled) {
    if (imp > th_h) return TIER_HI;
    if (c->mid_enabled && imp >= am / (float)n) return TIER_MID;
    if (imp >= th_l) return TIER_LO;
    return TIER_PRUNE;
  }
  return imp >= th_l ? TIER_HI : TIER_PRUNE;
}

/* precision order of the levels: prune < lo < mid < hi */
static int tier_rank(int tier) {
  return tier == TIER_HI ? 3 : tier == TIER_MID ? 2 : tier == TIER_LO ? 1 : 0;
}

/* Prompt scores of one KV head, fp64. Compaction policy, prompt phase: the
 * importance of token j is the mean of the attention it receives from later
 * queries (here the last 32 prompt positions), with the heads of a GQA group
 * combined by max. S_j = sum over observation queries p >= j of
 * max_h softmax_j(q_{h,p} . k / sqrt(d)) over keys j' <= p. */
void orc_unit_scores(int n0, int G, const uint16_t* k, int64_t k_stride, const uint16_t* q,
                     int64_t q_obs_stride, int64_t q_head_stride, double* S) {
  double* kd = (double*)malloc(sizeof(double) * (size_t)n0 * D);
  double* logit = (double*)malloc(sizeof(double) * (size_t)n0);
  double* pmax = (double*)malloc(sizeof(double) * (size_t)n0);
  for (int64_t j = 0; j < n0; j++)
    for (int f = 0; f < D; f++) kd[j * D + f] = orc_half_to_float(k[j * k_stride + f]);
  const double scale = 1.0 / sqrt((double)D);
  for (int j = 0; j < n0; j++) S[j] = 0.0;
  for (int o = 0; o < OBS; o++) {
    int p = n0 - OBS + o;
    if (p < 0) continue;
    for (int j = 0; j <= p; j++) pmax[j] = 0.0;
    for (int h = 0; h < G; h++) {
      double qd[D];
      for (int f = 0; f < D; f++) qd[f] = orc_half_to_float(q[o * q_obs_stride + h * q_head_stride + f]);
      double m = -INFINITY;
      for (int j = 0; j <= p; j++) {
        double acc = 0.0;
        for (int f = 0; f < D; f++) acc += qd[f] * kd[(int64_t)j * D + f];
        logit[j] = acc * scale;
        if (logit[j] > m) m = logit[j];
      }
      double sum = 0.0;
      for (int j = 0; j <= p; j++) sum += exp(logit[j] - m);
      double lse = m + log(sum);
      for (int j = 0; j <= p; j++) {
        double pj = exp(logit[j] - lse);
        if (pj > pmax[j]) pmax[j] = pj;
      }
    }
    for (int j = 0; j <= p; j++) S[j] += pmax[j];
  }
  free(kd); free(logit); free(pmax);
}

/* Causal prefill attention of one KV head's G query heads, fp64 — the
 * model's own attention over the prompt, after which DiffKV's compactor runs
 * (System implementation, architecture overview; Background, attention
 * equation): out[p][h] = sum_{j <= p} softmax_j(q_{p,h} . k_j / sqrt(d)) v_j,
 * and lse2[p][h] = log2 sum_{j <= p} exp(q_{p,h} . k_j / sqrt(d)), the
 * log-sum-exp in base 2 that the score pass of the prompt compaction uses.
 * One query row qd (D doubles) at position p over keys kd / vd (rows of D
 * doubles); w holds p + 1 doubles of work space. */
static void prefill_row(int p, const double* qd, const double* kd, const double* vd, double* w, double* o,
                        double* lse2) {
  const double scale = 1.0 / sqrt((double)D);
  double m = -INFINITY;
  for (int j = 0; j <= p; j++) {
    double acc = 0.0;
    for (int f = 0; f < D; f++) acc += qd[f] * kd[(int64_t)j * D + f];
    w[j] = acc * scale;
    if (w[j] > m) m = w[j];
  }
  double sum = 0.0;
  for (int j = 0; j <= p; j++) {
    w[j] = exp(w[j] - m);
    sum += w[j];
  }
  for (int f = 0; f < D; f++) o[f] = 0.0;
  for (int j = 0; j <= p; j++)
    for (int f = 0; f < D; f++) o[f] += w[j] * vd[(int64_t)j * D + f];
  for (int f = 0; f < D; f++) o[f] /= sum;
  *lse2 = (m + log(sum)) / log(2.0);
}

static void widen_rows(int n, const uint16_t* x, int64_t stride, double* xd) {
  for (int64_t j = 0; j < n; j++)
    for (int f = 0; f < D; f++) xd[j * D + f] = orc_half_to_float(x[j * stride + f]);
}

/* Every row of a prompt of n0 tokens: q rows are q + p * q_stride + h * D,
 * k / v rows k + j * kv_stride; out [n0][G][D], lse2 [n0][G]. */
void orc_prefill_attention(int n0, int G, const uint16_t* q, int64_t q_stride, const uint16_t* k,
                           const uint16_t* v, int64_t kv_stride, double* out, double* lse2) {
  double* kd = (double*)malloc(sizeof(double) * (size_t)n0 * D);
  double* vd = (double*)malloc(sizeof(double) * (size_t)n0 * D);
  double* w = (double*)malloc(sizeof(double) * (size_t)n0);
  widen_rows(n0, k, kv_stride, kd);
  widen_rows(n0, v, kv_stride, vd);
  for (int p = 0; p < n0; p++)
    for (int h = 0; h < G; h++) {
      double qd[D];
      for (int f = 0; f < D; f++) qd[f] = orc_half_to_float(q[(int64_t)p * q_stride + (int64_t)h * D + f]);
      prefill_row(p, qd, kd, vd, w, out + ((int64_t)p * G + h) * D, lse2 + (int64_t)p * G + h);
    }
  free(kd); free(vd); free(w);
}

/* Selected rows of the same attention: row r is the query at position
 * pos[r] (q + r * q_stride + h * D), over keys 0..pos[r] of k / v; out
 * [m][G][D], lse2 [m][G]. For checking single outputs of long prompts. */
void orc_prefill_rows(int m, int G, const int32_t* pos, const uint16_t* q, int64_t q_stride, const uint16_t* k,
                      const uint16_t* v, int64_t kv_stride, double* out, double* lse2) {
  int n = 0;
  for (int r = 0; r < m; r++)
    if (pos[r] + 1 > n) n = pos[r] + 1;
  double* kd = (double*)malloc(sizeof(double) * (size_t)n * D);
  double* vd = (double*)malloc(sizeof(double) * (size_t)n * D);
  double* w = (double*)malloc(sizeof(double) * (size_t)n);
  widen_rows(n, k, kv_stride, kd);
  widen_rows(n, v, kv_stride, vd);
  for (int r = 0; r < m; r++)
    for (int h = 0; h < G; h++) {
      double qd[D];
      for (int f = 0; f < D; f++) qd[f] = orc_half_to_float(q[(int64_t)r * q_stride + (int64_t)h * D + f]);
      prefill_row(pos[r], qd, kd, vd, w, out + ((int64_t)r * G + h) * D, lse2 + (int64_t)r * G + h);
    }
  free(kd); free(vd); free(w);
}

/* ------------------------------------------------------------------ */
/* Prompt phase — Memory management, prompt workflow (Figure 6).       */
/* ------------------------------------------------------------------ */
int orc_prompt_step(orc_pool* p, int layer, int n_req, const int32_t* slots, const int32_t* lens,
                    const uint16_t* k, const uint16_t* v, const uint16_t* q_obs,
                    const float* scores_in, float* scores_out) {
  const orc_config* c = &p->c;
  const int H = c->n_kv_heads, G = c->group_size, Hq = H * G;
  const int th = p->tg[TIER_HI].t, tl = p->tg[TIER_LO].t, tm = p->tg[TIER_MID].t;
  if (layer < 0 || layer >= c->n_layers || n_req < 1 || n_req > c->max_requests) return ORC_ERR_ARG;
  for (int i = 0; i < n_req; i++) {
    if (slots[i] < 0 || slots[i] >= c->max_requests) return ORC_ERR_ARG;
    if (lens[i] < 1 || lens[i] > c->max_seq_len) return ORC_ERR_ARG;
    for (int j = 0; j < i; j++) if (slots[j] == slots[i]) return ORC_ERR_ARG;
    if (rstate(p, layer, slots[i])[0]) return ORC_ERR_STATE;
  }
  if (!scores_in && !q_obs) return ORC_ERR_ARG;
  const int nh = n_req * H;
  int64_t* tok0 = (int64_t*)malloc(sizeof(int64_t) * (n_req + 1));
  tok0[0] = 0;
  for (int i = 0; i < n_req; i++) tok0[i + 1] = tok0[i] + lens[i];

  /* conservative grant: every head assumes all tokens hi (plus slack) */
  int* grant = (int*)malloc(sizeof(int) * nh);
  int64_t total = 0;
  for (int i = 0; i < n_req; i++)
    for (int h = 0; h < H; h++) {
      grant[i * H + h] = (lens[i] + th - 1) / th + c->grant_slack;
      total += grant[i * H + h];
    }
  if (total > p->ptr[1] - p->ptr[0]) { free(tok0); free(grant); return ORC_ERR_NO_PAGES; }

  /* planning: every head scores and classifies its tokens independently */
  float* S32 = (float*)malloc(sizeof(float) * (size_t)tok0[n_req] * H);
  uint8_t* tier = (uint8_t*)malloc((size_t)tok0[n_req] * H);
  int* nhi = (int*)calloc(nh, sizeof(int));
  int* nlo = (int*)calloc(nh, sizeof(int));
  int* nmid = (int*)calloc(nh, sizeof(int));
  int status = ORC_OK;
  for (int i = 0; i < n_req && status == ORC_OK; i++) {
    const int n0 = lens[i];
    double* S = (double*)malloc(sizeof(double) * (size_t)n0);
    for (int h = 0; h < H; h++) {
      if (scores_in) {
        for (int j = 0; j < n0; j++) S[j] = scores_in[(tok0[i] + j) * H + h];
      } else {
        orc_unit_scores(n0, G, k + (tok0[i] * H + h) * D, (int64_t)H * D,
                        q_obs + ((int64_t)i * OBS * Hq + (int64_t)h * G) * D, (int64_t)Hq * D, D, S);
      }
      const size_t hx = (size_t)layer * H + h;
      for (int j = 0; j < n0; j++) {
        int64_t t = (tok0[i] + j) * H + h;
        float s32 = (float)S[j];
        S32[t] = s32;
        int tr;
        if (j >= n0 - c->window) tr = TIER_HI;            /* recent window */
        else tr = classify(c, p->alpha + 2 * hx, p->alpha_mid[hx], importance(s32, score_count(j, n0, 0)), n0);
        tier[t] = (uint8_t)tr;
        if (tr == TIER_HI) nhi[i * H + h]++;
        else if (tr == TIER_LO) nlo[i * H + h]++;
        else if (tr == TIER_MID) nmid[i * H + h]++;
      }
      int php = (nhi[i * H + h] + th - 1) / th, plp = (nlo[i * H + h] + tl - 1) / tl;
      int pmp = (nmid[i * H + h] + tm - 1) / tm;
      if (php + pmp + plp > grant[i * H + h] || php + plp > p->table_len || pmp > p->mid_len)
        status = ORC_ERR_TABLE_FULL;
    }
    free(S);
  }
  if (status != ORC_OK) {
    free(tok0); free(grant); free(S32); free(tier); free(nhi); free(nlo); free(nmid);
    return status;
  }

  /* coordination 1: exclusive prefix sum of grants at the list start */
  int** gp = (int**)malloc(sizeof(int*) * nh);
  int64_t off = 0;
  for (int hd = 0; hd < nh; hd++) {
    gp[hd] = (int*)malloc(sizeof(int) * grant[hd]);
    for (int x = 0; x < grant[hd]; x++) gp[hd][x] = p->list[(p->ptr[0] + off + x) % c->n_pages];
    off += grant[hd];
  }

  /* pack: hi tokens fill the grant from the left, lo tokens from the right,
   * mid tokens (third level) the grant pages after the hi ones */
  for (int i = 0; i < n_req; i++) {
    const int n0 = lens[i];
    for (int h = 0; h < H; h++) {
      int hd = i * H + h, rh = 0, rl = 0, rm = 0;
      const int php = (nhi[hd] + th - 1) / th;
      for (int j = 0; j < n0; j++) {
        int64_t t = (tok0[i] + j) * H + h;
        if (tier[t] == TIER_PRUNE) continue;
        float kx[D], vx[D];
        half_vec(k + t * D, kx);
        half_vec(v + t * D, vx);
        token_rec r;
        make_token(kx, vx, &p->tg[tier[t]], S32[t], j, &r);
        if (tier[t] == TIER_HI) {
          put_token(page_ptr(p, gp[hd][rh / th]), &p->tg[TIER_HI], rh % th, &r);
          rh++;
        } else if (tier[t] == TIER_LO) {
          put_token(page_ptr(p, gp[hd][grant[hd] - 1 - rl / tl]), &p->tg[TIER_LO], rl % tl, &r);
          rl++;
        } else {
          put_token(page_ptr(p, gp[hd][php + rm / tm]), &p->tg[TIER_MID], rm % tm, &r);
          rm++;
        }
      }
    }
  }

  /* coordination 2: exclusive prefix sum of unused middle pages at the list end;
   * the bidirectional table records hi pages from the left, lo from the right,
   * and its one-way part the mid pages */
  int64_t roff = 0;
  for (int i = 0; i < n_req; i++)
    for (int h = 0; h < H; h++) {
      int hd = i * H + h;
      int php = (nhi[hd] + th - 1) / th, plp = (nlo[hd] + tl - 1) / tl, pmp = (nmid[hd] + tm - 1) / tm;
      for (int x = php + pmp; x < grant[hd] - plp; x++) {
        p->list[(p->ptr[1] + roff) % c->n_pages] = gp[hd][x];
        roff++;
      }
      int32_t* row = trow(p, layer, slots[i], h);
      for (int e = 0; e < p->row_len; e++) row[e] = -1;
      for (int x = 0; x < php; x++) row[x] = gp[hd][x];
      for (int x = 0; x < plp; x++) row[p->table_len - 1 - x] = gp[hd][grant[hd] - 1 - x];
      for (int x = 0; x < pmp; x++) row[p->table_len + x] = gp[hd][php + x];
      int32_t* cn = hcnt(p, layer, slots[i], h);
      cn[0] = nhi[hd]; cn[1] = nlo[hd]; cn[2] = php; cn[3] = plp;
      if (c->mid_enabled) { cn[4] = nmid[hd]; cn[5] = pmp; }
    }
  p->ptr[0] += total;
  p->ptr[1] += roff;
  for (int i = 0; i < n_req; i++) {
    int32_t* rs = rstate(p, layer, slots[i]);
    rs[0] = 1; rs[1] = lens[i]; rs[2] = lens[i]; rs[3] = 0;
  }
  if (scores_out) memcpy(scores_out, S32, sizeof(float) * (size_t)tok0[n_req] * H);
  for (int hd = 0; hd < nh; hd++) free(gp[hd]);
  free(gp); free(tok0); free(grant); free(S32); free(tier); free(nhi); free(nlo); free(nmid);
  return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Generation phase — Compaction policy (generation phase, algorithm   */
/* flow) and Memory management (generation workflow).                 */
/* ------------------------------------------------------------------ */

/* A slot's content after the step, described by where it comes from: a
 * token stored before the step (its tier and slot then), or the new token. */
enum { SRC_STORED = 0, SRC_NEW = 1 };
typedef struct { int kind, tier, slot; float imp; int pos; } src_t;

/* the levels a head can hold, in the order of their page allocations */
static const int k_tiers[3] = {TIER_HI, TIER_LO, TIER_MID};

typedef struct {
  src_t* a[4]; int n[4];                   /* slots of each tier after the step */
  int np[4], newp[4], freep[4];            /* page counts after, new and freed pages */
} head_plan;

static void remove_at(src_t* a, int* n, int x) {   /* swap-with-last */
  a[x] = a[*n - 1];
  (*n)--;
}

/* argmin of importance, ties to the smallest position; only entries whose
 * position is below `limit` are eligible; -1 if none */
static int argmin_imp(const src_t* a, int n, int limit) {
  int best = -1;
  for (int x = 0; x < n; x++) {
    if (a[x].pos >= limit) continue;
    if (best < 0 || a[x].imp < a[best].imp || (a[x].imp == a[best].imp && a[x].pos < a[best].pos))
      best = x;
  }
  return best;
}

/* ints of per-tier counters in a head's counter row: tokens, pages */
static int cnt_tok(int tier) { return tier == TIER_HI ? 0 : tier == TIER_LO ? 1 : 4; }
static int cnt_pg(int tier) { return tier == TIER_HI ? 2 : tier == TIER_LO ? 3 : 5; }
/* table entry of page k of a tier */
static int tab_entry(const orc_pool* p, int tier, int k) {
  return tier == TIER_HI ? k : tier == TIER_LO ? p->table_len - 1 - k : p->table_len + k;
}

int orc_decode_step(orc_pool* p, int layer, int n_req, const int32_t* slots, const uint16_t* k,
                    const uint16_t* v) {
  const orc_config* c = &p->c;
  const int H = c->n_kv_heads, L = p->table_len;
  const int ntiers = c->mid_enabled ? 3 : 2;
  if (layer < 0 || layer >= c->n_layers || n_req < 1 || n_req > c->max_requests) return ORC_ERR_ARG;
  /* generation-phase compaction needs a recent window of at least one token,
   * so that the newest token is never its own candidate */
  if (c->window < 1) return ORC_ERR_ARG;
  for (int i = 0; i < n_req; i++) {
    if (slots[i] < 0 || slots[i] >= c->max_requests) return ORC_ERR_ARG;
    for (int j = 0; j < i; j++) if (slots[j] == slots[i]) return ORC_ERR_ARG;
    int32_t* rs = rstate(p, layer, slots[i]);
    if (!rs[0]) return ORC_ERR_STATE;
    if (rs[2] + 1 > c->max_seq_len) return ORC_ERR_ARG;
  }
  const int nh = n_req * H;
  head_plan* pl = (head_plan*)calloc(nh, sizeof(head_plan));
  int64_t need = 0;
  int status = ORC_OK;
  for (int i = 0; i < n_req; i++) {
    int32_t* rs = rstate(p, layer, slots[i]);
    const int n0 = rs[1], n = rs[2] + 1, upd = rs[3];
    for (int h = 0; h < H; h++) {
      const size_t hx = (size_t)layer * H + h;
      const float* alpha = p->alpha + 2 * hx;
      const float am = p->alpha_mid[hx];
      head_plan* q = &pl[i * H + h];
      int32_t* cn = hcnt(p, layer, slots[i], h);
      int32_t* row = trow(p, layer, slots[i], h);
      for (int x = 0; x < ntiers; x++) {
        const int tier = k_tiers[x], cnt = cn[cnt_tok(tier)];
        const tier_geom* g = &p->tg[tier];
        src_t* a = q->a[tier] = (src_t*)malloc(sizeof(src_t) * (cnt + 2));
        q->n[tier] = cnt;
        for (int s = 0; s < cnt; s++) {
          int ip;
          const uint8_t* pg = slot_loc(p, row, tier, s, &ip);
          float sc; int32_t pos;
          memcpy(&sc, pg + g->off[4] + 4 * ip, 4);
          memcpy(&pos, pg + g->off[5] + 4 * ip, 4);
          a[s].kind = SRC_STORED; a[s].tier = tier; a[s].slot = s; a[s].pos = pos;
          a[s].imp = importance(sc, score_count(pos, n0, upd));
        }
      }
      src_t* hi = q->a[TIER_HI];
      /* (1) the newest token enters the recent window at high precision */
      src_t nw = {SRC_NEW, TIER_HI, -1, 0.0f, n - 1};
      hi[q->n[TIER_HI]++] = nw;
      /* (2) the window's oldest token t_c leaves it and is classified */
      const int pc = n - c->window - 1;
      if (pc >= 0) {
        int xc = -1;
        for (int x = 0; x < q->n[TIER_HI]; x++) if (hi[x].pos == pc) { xc = x; break; }
        if (xc < 0) { status = ORC_ERR_CHECK; }
        else {
          const int tc = classify(c, alpha, am, hi[xc].imp, n);
          int vt;                                   /* tier whose victim is considered */
          if (tc == TIER_HI) {
            vt = TIER_HI;                           /* t_c stays hi */
          } else if (tc == TIER_PRUNE) {
            vt = -1;
            remove_at(hi, &q->n[TIER_HI], xc);
          } else {                                  /* t_c moves to its lower level */
            src_t t = hi[xc];
            remove_at(hi, &q->n[TIER_HI], xc);
            q->a[tc][q->n[tc]++] = t;
            vt = tc;
          }
          /* (3) the victim: the least important token of the level t_c ended
           * in (hi: outside the window; t_c itself is eligible), kept if it
           * still classifies at that level or above, else moved to the level
           * it classifies at, or pruned */
          if (vt >= 0) {
            src_t* a = q->a[vt];
            const int xv = argmin_imp(a, q->n[vt], vt == TIER_HI ? n - c->window : 0x7fffffff);
            const int cv = classify(c, alpha, am, a[xv].imp, n);
            if (tier_rank(cv) < tier_rank(vt)) {
              src_t t = a[xv];
              remove_at(a, &q->n[vt], xv);
              if (cv != TIER_PRUNE) q->a[cv][q->n[cv]++] = t;
            }
          }
        }
      }
      /* page need of the step, from the net change of each tier */
      for (int x = 0; x < ntiers; x++) {
        const int tier = k_tiers[x], t = p->tg[tier].t;
        const int pneed = (q->n[tier] + t - 1) / t, p0 = cn[cnt_pg(tier)];
        q->np[tier] = p0;
        if (pneed > p0) { q->newp[tier] = pneed - p0; q->np[tier] = pneed; }
        else if (c->reclaim_in_decode && pneed < p0) { q->freep[tier] = p0 - pneed; q->np[tier] = pneed; }
        need += q->newp[tier];
      }
      if (status == ORC_OK &&
          (q->np[TIER_HI] + q->np[TIER_LO] > L || (c->mid_enabled && q->np[TIER_MID] > p->mid_len)))
        status = ORC_ERR_TABLE_FULL;
    }
  }
  if (status == ORC_OK && need > p->ptr[1] - p->ptr[0]) status = ORC_ERR_NO_PAGES;
  if (status != ORC_OK) {
    for (int hd = 0; hd < nh; hd++) for (int x = 0; x < ntiers; x++) free(pl[hd].a[k_tiers[x]]);
    free(pl);
    return status;
  }
  /* commit: new pages by one prefix sum at the list start (per head hi, lo,
   * then mid), emptied tail pages by one at the list end (same order) */
  int64_t aoff = 0, roff = 0;
  for (int i = 0; i < n_req; i++) {
    int32_t* rs = rstate(p, layer, slots[i]);
    const int n = rs[2] + 1;
    for (int h = 0; h < H; h++) {
      head_plan* q = &pl[i * H + h];
      int32_t* cn = hcnt(p, layer, slots[i], h);
      int32_t* row = trow(p, layer, slots[i], h);
      /* read every source record from the state before the step */
      token_rec* recs[4] = {0, 0, 0, 0};
      int* dirty[4] = {0, 0, 0, 0};
      for (int y = 0; y < ntiers; y++) {
        const int tier = k_tiers[y];
        recs[tier] = (token_rec*)malloc(sizeof(token_rec) * (q->n[tier] + 1));
        dirty[tier] = (int*)calloc(q->n[tier] + 1, sizeof(int));
        for (int x = 0; x < q->n[tier]; x++) {
          src_t s = q->a[tier][x];
          if (s.kind == SRC_STORED && s.tier == tier && s.slot == x) continue;   /* unchanged */
          dirty[tier][x] = 1;
          if (s.kind == SRC_NEW) {
            float kx[D], vx[D];
            half_vec(k + ((int64_t)i * H + h) * D, kx);
            half_vec(v + ((int64_t)i * H + h) * D, vx);
            make_token(kx, vx, &p->tg[TIER_HI], 0.0f, n - 1, &recs[tier][x]);
          } else {
            int ip;
            token_rec t;
            const uint8_t* pg = slot_loc(p, row, s.tier, s.slot, &ip);
            get_token(pg, &p->tg[s.tier], ip, &t);
            if (s.tier == tier) recs[tier][x] = t;                  /* moved inside its level */
            else requant(&t, &p->tg[tier], &recs[tier][x]);        /* to a lower level */
          }
        }
      }
      /* allocate, then free, then write */
      for (int y = 0; y < ntiers; y++) {
        const int tier = k_tiers[y];
        for (int x = 0; x < q->newp[tier]; x++)
          row[tab_entry(p, tier, cn[cnt_pg(tier)] + x)] = p->list[(p->ptr[0] + aoff++) % c->n_pages];
      }
      for (int y = 0; y < ntiers; y++) {
        const int tier = k_tiers[y];
        for (int x = 0; x < q->freep[tier]; x++) {
          int e = tab_entry(p, tier, cn[cnt_pg(tier)] - 1 - x);
          p->list[(p->ptr[1] + roff++) % c->n_pages] = row[e];
          row[e] = -1;
        }
      }
      for (int y = 0; y < ntiers; y++) {
        const int tier = k_tiers[y];
        for (int x = 0; x < q->n[tier]; x++) {
          if (!dirty[tier][x]) continue;
          int ip;
          uint8_t* pg = slot_loc(p, row, tier, x, &ip);
          put_token(pg, &p->tg[tier], ip, &recs[tier][x]);
        }
        cn[cnt_tok(tier)] = q->n[tier];
        cn[cnt_pg(tier)] = q->np[tier];
        free(recs[tier]); free(dirty[tier]);
      }
    }
    rs[2] = n;
  }
  p->ptr[0] += aoff;
  p->ptr[1] += roff;
  for (int hd = 0; hd < nh; hd++) for (int x = 0; x < ntiers; x++) free(pl[hd].a[k_tiers[x]]);
  free(pl);
  return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Decode attention — Background, attention equation, over the         */
/* dequantized mixed-precision pages (hi pages first, then lo).        */
/* ------------------------------------------------------------------ */

/* Stored token j of a head in attention order (hi slots, then mid slots,
 * then lo slots): its tier and slot. cn: the head's counters; nm: its mid
 * tokens (0 without the mid level). */
static void stored_index(const int32_t* cn, int nm, int j, int* tier, int* s) {
  if (j < cn[0]) { *tier = TIER_HI; *s = j; }
  else if (j < cn[0] + nm) { *tier = TIER_MID; *s = j - cn[0]; }
  else { *tier = TIER_LO; *s = j - cn[0] - nm; }
}

/* Attention of one KV head's G query heads (q: G x 128 fp16, contiguous)
 * over its stored tokens; out: G x 128 fp64; if pmax is non-NULL it
 * receives, per stored token (hi slots then lo slots), the max over the G
 * heads of its softmax probability. Returns the number of stored tokens. */
int orc_unit_attention(orc_pool* p, int layer, int slot, int kvh, const uint16_t* q, double* out,
                       double* pmax) {
  const int G = p->c.group_size;
  int32_t* cn = hcnt(p, layer, slot, kvh);
  int32_t* row = trow(p, layer, slot, kvh);
  const int nm = p->c.mid_enabled ? cn[4] : 0;
  const int n = cn[0] + nm + cn[1];
  double* kh = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * D);
  double* vh = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * D);
  for (int j = 0; j < n; j++) {
    int tier, s;
    stored_index(cn, nm, j, &tier, &s);
    token_rec r;
    int ip;
    const uint8_t* pg = slot_loc(p, row, tier, s, &ip);
    get_token(pg, &p->tg[tier], ip, &r);
    double ks = orc_half_to_float(r.ks), kz = orc_half_to_float(r.kz);
    double vs = orc_half_to_float(r.vs), vz = orc_half_to_float(r.vz);
    for (int f = 0; f < D; f++) {
      kh[(int64_t)j * D + f] = ks * r.kc[f] + kz;     /* exact in fp64 */
      vh[(int64_t)j * D + f] = vs * r.vc[f] + vz;
    }
  }
  double* l = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  if (pmax) for (int j = 0; j < n; j++) pmax[j] = 0.0;
  const double scale = 1.0 / sqrt((double)D);
  for (int h = 0; h < G; h++) {
    double qd[D];
    for (int f = 0; f < D; f++) qd[f] = orc_half_to_float(q[h * D + f]);
    double m = -INFINITY;
    for (int j = 0; j < n; j++) {
      double acc = 0.0;
      for (int f = 0; f < D; f++) acc += qd[f] * kh[(int64_t)j * D + f];
      l[j] = acc * scale;
      if (l[j] > m) m = l[j];
    }
    double sum = 0.0;
    for (int j = 0; j < n; j++) sum += exp(l[j] - m);
    for (int f = 0; f < D; f++) out[h * D + f] = 0.0;
    for (int j = 0; j < n; j++) {
      double pj = exp(l[j] - m) / sum;
      for (int f = 0; f < D; f++) out[h * D + f] += pj * vh[(int64_t)j * D + f];
      if (pmax && pj > pmax[j]) pmax[j] = pj;
    }
  }
  free(kh); free(vh); free(l);
  return n;
}

int orc_decode_attention(orc_pool* p, int layer, int n_req, const int32_t* slots, const uint16_t* q,
                         double* out, int update_scores) {
  const int H = p->c.n_kv_heads, G = p->c.group_size;
  if (layer < 0 || layer >= p->c.n_layers || n_req < 1) return ORC_ERR_ARG;
  for (int i = 0; i < n_req; i++) {
    if (slots[i] < 0 || slots[i] >= p->c.max_requests) return ORC_ERR_ARG;
    if (!rstate(p, layer, slots[i])[0]) return ORC_ERR_STATE;
  }
  for (int i = 0; i < n_req; i++) {
    for (int h = 0; h < H; h++) {
      int32_t* cn = hcnt(p, layer, slots[i], h);
      int32_t* row = trow(p, layer, slots[i], h);
      const int nm = p->c.mid_enabled ? cn[4] : 0;
      int n = cn[0] + nm + cn[1];
      double* pm = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
      orc_unit_attention(p, layer, slots[i], h, q + ((int64_t)i * H * G + (int64_t)h * G) * D,
                         out + ((int64_t)i * H * G + (int64_t)h * G) * D, pm);
      if (update_scores) {
        for (int j = 0; j < n; j++) {
          int tier, s;
          stored_index(cn, nm, j, &tier, &s);
          const tier_geom* g = &p->tg[tier];
          int ip;
          uint8_t* sp = slot_loc(p, row, tier, s, &ip) + g->off[4] + 4 * ip;
          float sc;
          memcpy(&sc, sp, 4);
          sc = (float)((double)sc + pm[j]);
          memcpy(sp, &sc, 4);
        }
      }
      free(pm);
    }
    if (update_scores) rstate(p, layer, slots[i])[3] += 1;
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Request completion — Memory management, generation workflow: all    */
/* pages of a finished request are reclaimed.                          */
/* ------------------------------------------------------------------ */
int orc_free_request(orc_pool* p, int slot) {
  const orc_config* c = &p->c;
  if (slot < 0 || slot >= c->max_requests) return ORC_ERR_ARG;
  int any = 0;
  for (int l = 0; l < c->n_layers; l++) any |= rstate(p, l, slot)[0];
  if (!any) return ORC_ERR_STATE;
  for (int l = 0; l < c->n_layers; l++) {
    for (int h = 0; h < c->n_kv_heads; h++) {
      int32_t* cn = hcnt(p, l, slot, h);
      int32_t* row = trow(p, l, slot, h);
      for (int x = 0; x < cn[2]; x++) p->list[(p->ptr[1]++) % c->n_pages] = row[x];
      for (int x = 0; x < cn[3]; x++) p->list[(p->ptr[1]++) % c->n_pages] = row[p->table_len - 1 - x];
      if (c->mid_enabled)
        for (int x = 0; x < cn[5]; x++) p->list[(p->ptr[1]++) % c->n_pages] = row[p->table_len + x];
      for (int e = 0; e < p->row_len; e++) row[e] = -1;
      for (int x = 0; x < p->cstride; x++) cn[x] = 0;
    }
    int32_t* rs = rstate(p, l, slot);
    rs[0] = rs[1] = rs[2] = rs[3] = 0;
  }
  return ORC_OK;
}
