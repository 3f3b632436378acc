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
} orc_config;

typedef struct {
  int t;                       /* tokens per page */
  int kbits, vbits, g;         /* g = tokens sharing one value byte */
  int off[6];                  /* K codes, V codes, K meta, V meta, score, position */
  int used;
} tier_geom;

typedef struct {
  orc_config c;
  tier_geom tg[3];             /* indexed by TIER_LO / TIER_HI */
  int table_len;
  uint8_t* pages;
  int32_t* list;
  int64_t ptr[2];              /* start, end */
  int32_t* table;              /* [layer][slot][kvh][table_len] */
  int32_t* counts;             /* [layer][slot][kvh][4] hi tok, lo tok, hi pages, lo pages */
  int32_t* req;                /* [layer][slot][4] active, N0, N, updates */
  float* alpha;                /* [layer][kvh][2] alpha_h, alpha_l of each head */
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
  return p->table + (((int64_t)layer * p->c.max_requests + slot) * p->c.n_kv_heads + kvh) * p->table_len;
}
static int32_t* hcnt(orc_pool* p, int layer, int slot, int kvh) {
  return p->counts + (((int64_t)layer * p->c.max_requests + slot) * p->c.n_kv_heads + kvh) * 4;
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
  int th = c->t_hi ? c->t_hi : fit_tokens(&p->tg[TIER_HI], c->page_bytes);
  int tl = c->t_lo ? c->t_lo : fit_tokens(&p->tg[TIER_LO], c->page_bytes);
  layout(&p->tg[TIER_HI], th);
  layout(&p->tg[TIER_LO], tl);
  /* Bidirectional page table entry length: max sequence length over tokens per
   * hi page, plus one page for a hi/lo split whose two partial pages exceed it. */
  p->table_len = (c->max_seq_len + th - 1) / th + 1;
  p->pages = (uint8_t*)calloc((size_t)c->n_pages, (size_t)c->page_bytes);
  p->list = (int32_t*)malloc(sizeof(int32_t) * (size_t)c->n_pages);
  for (int i = 0; i < c->n_pages; i++) p->list[i] = i;
  p->ptr[0] = 0;
  p->ptr[1] = c->n_pages;
  size_t heads = (size_t)c->n_layers * c->max_requests * c->n_kv_heads;
  p->table = (int32_t*)malloc(sizeof(int32_t) * heads * p->table_len);
  for (size_t i = 0; i < heads * p->table_len; i++) p->table[i] = -1;
  p->counts = (int32_t*)calloc(heads * 4, sizeof(int32_t));
  p->req = (int32_t*)calloc((size_t)c->n_layers * c->max_requests * 4, sizeof(int32_t));
  /* every head starts with the configuration's thresholds */
  p->alpha = (float*)malloc(sizeof(float) * 2 * (size_t)c->n_layers * c->n_kv_heads);
  for (int x = 0; x < c->n_layers * c->n_kv_heads; x++) {
    p->alpha[2 * x] = c->alpha_h;
    p->alpha[2 * x + 1] = c->alpha_l;
  }
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

void orc_pool_free(orc_pool* p) {
  if (!p) return;
  free(p->pages); free(p->list); free(p->table); free(p->counts); free(p->req); free(p->alpha);
  free(p);
}

/* geometry: t_hi, t_lo, table_len, hi off[6], lo off[6], hi used, lo used */
void orc_geometry(const orc_pool* p, int32_t* out) {
  out[0] = p->tg[TIER_HI].t;
  out[1] = p->tg[TIER_LO].t;
  out[2] = p->table_len;
  for (int i = 0; i < 6; i++) out[3 + i] = p->tg[TIER_HI].off[i];
  for (int i = 0; i < 6; i++) out[9 + i] = p->tg[TIER_LO].off[i];
  out[15] = p->tg[TIER_HI].used;
  out[16] = p->tg[TIER_LO].used;
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

/* hi -> lo re-quantization of a stored token: dequantize, quantize again */
static void demote(const token_rec* hi, const tier_geom* lo, token_rec* out) {
  float k[D], v[D];
  for (int f = 0; f < D; f++) {
    k[f] = orc_dequant(hi->ks, hi->kz, hi->kc[f]);
    v[f] = orc_dequant(hi->vs, hi->vz, hi->vc[f]);
  }
  make_token(k, v, lo, hi->score, hi->pos, out);
}

/* page holding slot s of a tier (through the bidirectional table row) and
 * the slot's index inside that page */
static uint8_t* slot_loc(orc_pool* p, const int32_t* row, int tier, int s, int* in_page) {
  const int t = p->tg[tier].t;
  *in_page = s % t;
  int e = tier == TIER_HI ? s / t : p->table_len - 1 - s / t;
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
 * with the lo tier disabled a token that would be lo is kept at hi precision */
static int classify(const orc_config* c, const float* alpha, float imp, int n) {
  float th_h = alpha[0] / (float)n, th_l = alpha[1] / (float)n;
  if (c->lo_enabled) {
    if (imp > th_h) return TIER_HI;
    if (imp >= th_l) return TIER_LO;
    return TIER_PRUNE;
  }
  return imp >= th_l ? TIER_HI : TIER_PRUNE;
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
  const int th = p->tg[TIER_HI].t, tl = p->tg[TIER_LO].t;
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
      for (int j = 0; j < n0; j++) {
        int64_t t = (tok0[i] + j) * H + h;
        float s32 = (float)S[j];
        S32[t] = s32;
        int tr;
        if (j >= n0 - c->window) tr = TIER_HI;            /* recent window */
        else tr = classify(c, p->alpha + 2 * ((size_t)layer * H + h), importance(s32, score_count(j, n0, 0)), n0);
        tier[t] = (uint8_t)tr;
        if (tr == TIER_HI) nhi[i * H + h]++;
        else if (tr == TIER_LO) nlo[i * H + h]++;
      }
      int php = (nhi[i * H + h] + th - 1) / th, plp = (nlo[i * H + h] + tl - 1) / tl;
      if (php + plp > grant[i * H + h] || php + plp > p->table_len) status = ORC_ERR_TABLE_FULL;
    }
    free(S);
  }
  if (status != ORC_OK) {
    free(tok0); free(grant); free(S32); free(tier); free(nhi); free(nlo);
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

  /* pack: hi tokens fill the grant from the left, lo tokens from the right */
  for (int i = 0; i < n_req; i++) {
    const int n0 = lens[i];
    for (int h = 0; h < H; h++) {
      int hd = i * H + h, rh = 0, rl = 0;
      for (int j = 0; j < n0; j++) {
        int64_t t = (tok0[i] + j) * H + h;
        if (tier[t] == TIER_PRUNE) continue;
        float kx[D], vx[D];
        half_vec(k + t * D, kx);
        half_vec(v + t * D, vx);
        token_rec r;
        if (tier[t] == TIER_HI) {
          make_token(kx, vx, &p->tg[TIER_HI], S32[t], j, &r);
          put_token(page_ptr(p, gp[hd][rh / th]), &p->tg[TIER_HI], rh % th, &r);
          rh++;
        } else {
          make_token(kx, vx, &p->tg[TIER_LO], S32[t], j, &r);
          put_token(page_ptr(p, gp[hd][grant[hd] - 1 - rl / tl]), &p->tg[TIER_LO], rl % tl, &r);
          rl++;
        }
      }
    }
  }

  /* coordination 2: exclusive prefix sum of unused middle pages at the list end;
   * the bidirectional table records hi pages from the left, lo from the right */
  int64_t roff = 0;
  for (int i = 0; i < n_req; i++)
    for (int h = 0; h < H; h++) {
      int hd = i * H + h;
      int php = (nhi[hd] + th - 1) / th, plp = (nlo[hd] + tl - 1) / tl;
      for (int x = php; x < grant[hd] - plp; x++) {
        p->list[(p->ptr[1] + roff) % c->n_pages] = gp[hd][x];
        roff++;
      }
      int32_t* row = trow(p, layer, slots[i], h);
      for (int e = 0; e < p->table_len; e++) row[e] = -1;
      for (int x = 0; x < php; x++) row[x] = gp[hd][x];
      for (int x = 0; x < plp; x++) row[p->table_len - 1 - x] = gp[hd][grant[hd] - 1 - x];
      int32_t* cn = hcnt(p, layer, slots[i], h);
      cn[0] = nhi[hd]; cn[1] = nlo[hd]; cn[2] = php; cn[3] = plp;
    }
  p->ptr[0] += total;
  p->ptr[1] += roff;
  for (int i = 0; i < n_req; i++) {
    int32_t* rs = rstate(p, layer, slots[i]);
    rs[0] = 1; rs[1] = lens[i]; rs[2] = lens[i]; rs[3] = 0;
  }
  if (scores_out) memcpy(scores_out, S32, sizeof(float) * (size_t)tok0[n_req] * H);
  for (int hd = 0; hd < nh; hd++) free(gp[hd]);
  free(gp); free(tok0); free(grant); free(S32); free(tier); free(nhi); free(nlo);
  return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Generation phase — Compaction policy (generation phase, algorithm   */
/* flow) and Memory management (generation workflow).                 */
/* ------------------------------------------------------------------ */

/* A slot's content after the step, described by where it comes from. */
enum { SRC_HI = 0, SRC_LO = 1, SRC_NEW = 2, SRC_DEMOTED = 3 };
typedef struct { int kind, slot; float imp; int pos; } src_t;

typedef struct {
  src_t* hi; int nh, cap_h;
  src_t* lo; int nl, cap_l;
  int new_hp, new_lp, free_hp, free_lp;    /* page changes of this head */
  int php, plp;                            /* page counts after the step */
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

int orc_decode_step(orc_pool* p, int layer, int n_req, const int32_t* slots, const uint16_t* k,
                    const uint16_t* v) {
  const orc_config* c = &p->c;
  const int H = c->n_kv_heads;
  const int th = p->tg[TIER_HI].t, tl = p->tg[TIER_LO].t, L = p->table_len;
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
      const float* alpha = p->alpha + 2 * ((size_t)layer * H + h);
      const float th_h = alpha[0] / (float)n, th_l = alpha[1] / (float)n;
      head_plan* q = &pl[i * H + h];
      int32_t* cn = hcnt(p, layer, slots[i], h);
      int32_t* row = trow(p, layer, slots[i], h);
      q->cap_h = cn[0] + 2; q->cap_l = cn[1] + 2;
      q->hi = (src_t*)malloc(sizeof(src_t) * q->cap_h);
      q->lo = (src_t*)malloc(sizeof(src_t) * q->cap_l);
      q->nh = cn[0]; q->nl = cn[1];
      for (int tr = 0; tr < 2; tr++) {
        int tier = tr ? TIER_LO : TIER_HI, cnt = tr ? cn[1] : cn[0];
        src_t* a = tr ? q->lo : q->hi;
        for (int s = 0; s < cnt; s++) {
          const tier_geom* g = &p->tg[tier];
          int ip;
          const uint8_t* pg = slot_loc(p, row, tier, s, &ip);
          float sc; int32_t pos;
          memcpy(&sc, pg + g->off[4] + 4 * ip, 4);
          memcpy(&pos, pg + g->off[5] + 4 * ip, 4);
          a[s].kind = tr ? SRC_LO : SRC_HI; a[s].slot = s; a[s].pos = pos;
          a[s].imp = importance(sc, score_count(pos, n0, upd));
        }
      }
      /* (1) the newest token enters the recent window at high precision */
      q->hi[q->nh].kind = SRC_NEW; q->hi[q->nh].slot = -1; q->hi[q->nh].pos = n - 1;
      q->hi[q->nh].imp = 0.0f;
      q->nh++;
      /* (2) the window's oldest token t_c leaves it and is classified */
      const int pc = n - c->window - 1;
      if (pc >= 0) {
        int xc = -1;
        for (int x = 0; x < q->nh; x++) if (q->hi[x].pos == pc) { xc = x; break; }
        if (xc < 0) { status = ORC_ERR_CHECK; }
        else {
          int tc = classify(c, alpha, q->hi[xc].imp, n);
          if (tc == TIER_HI) {
            /* t_c stays hi; the least important hi token outside the window is the victim */
            int xv = argmin_imp(q->hi, q->nh, n - c->window);
            float iv = q->hi[xv].imp;
            int keep = c->lo_enabled ? (iv > th_h) : (iv >= th_l);
            if (!keep) {
              src_t t = q->hi[xv];
              remove_at(q->hi, &q->nh, xv);
              if (c->lo_enabled && iv >= th_l) {               /* re-quantize to lo */
                src_t d = t; d.kind = SRC_DEMOTED;
                q->lo[q->nl++] = d;
              }
            }
          } else if (tc == TIER_LO) {
            src_t t = q->hi[xc];
            remove_at(q->hi, &q->nh, xc);
            src_t d = t; d.kind = SRC_DEMOTED;
            q->lo[q->nl++] = d;
            /* the least important lo token is the victim; pruned below alpha_l/N */
            int xv = argmin_imp(q->lo, q->nl, 0x7fffffff);
            if (q->lo[xv].imp < th_l) remove_at(q->lo, &q->nl, xv);
          } else {
            remove_at(q->hi, &q->nh, xc);
          }
        }
      }
      /* page need of the step, from the net change of each tier */
      int hp_need = (q->nh + th - 1) / th, lp_need = (q->nl + tl - 1) / tl;
      q->php = cn[2]; q->plp = cn[3];
      if (hp_need > q->php) { q->new_hp = hp_need - q->php; q->php = hp_need; }
      else if (c->reclaim_in_decode && hp_need < q->php) { q->free_hp = q->php - hp_need; q->php = hp_need; }
      if (lp_need > q->plp) { q->new_lp = lp_need - q->plp; q->plp = lp_need; }
      else if (c->reclaim_in_decode && lp_need < q->plp) { q->free_lp = q->plp - lp_need; q->plp = lp_need; }
      if (q->php + q->plp > L && status == ORC_OK) status = ORC_ERR_TABLE_FULL;
      need += q->new_hp + q->new_lp;
    }
  }
  if (status == ORC_OK && need > p->ptr[1] - p->ptr[0]) status = ORC_ERR_NO_PAGES;
  if (status != ORC_OK) {
    for (int hd = 0; hd < nh; hd++) { free(pl[hd].hi); free(pl[hd].lo); }
    free(pl);
    return status;
  }
  /* commit: new pages by one prefix sum at the list start (per head hi then lo) */
  int64_t aoff = 0, roff = 0;
  for (int i = 0; i < n_req; i++) {
    int32_t* rs = rstate(p, layer, slots[i]);
    const int n = rs[2] + 1;
    for (int h = 0; h < H; h++) {
      head_plan* q = &pl[i * H + h];
      int32_t* cn = hcnt(p, layer, slots[i], h);
      int32_t* row = trow(p, layer, slots[i], h);
      /* read every source record from the state before the step */
      token_rec* hi_new = (token_rec*)malloc(sizeof(token_rec) * (q->nh + 1));
      token_rec* lo_new = (token_rec*)malloc(sizeof(token_rec) * (q->nl + 1));
      int* hi_dirty = (int*)calloc(q->nh + 1, sizeof(int));
      int* lo_dirty = (int*)calloc(q->nl + 1, sizeof(int));
      for (int x = 0; x < q->nh; x++) {
        src_t s = q->hi[x];
        if (s.kind == SRC_HI && s.slot == x) continue;      /* unchanged */
        hi_dirty[x] = 1;
        if (s.kind == SRC_NEW) {
          float kx[D], vx[D];
          half_vec(k + ((int64_t)i * H + h) * D, kx);
          half_vec(v + ((int64_t)i * H + h) * D, vx);
          make_token(kx, vx, &p->tg[TIER_HI], 0.0f, n - 1, &hi_new[x]);
        } else {
          int ip;
          const uint8_t* pg = slot_loc(p, row, TIER_HI, s.slot, &ip);
          get_token(pg, &p->tg[TIER_HI], ip, &hi_new[x]);
        }
      }
      for (int x = 0; x < q->nl; x++) {
        src_t s = q->lo[x];
        if (s.kind == SRC_LO && s.slot == x) continue;
        lo_dirty[x] = 1;
        int ip;
        if (s.kind == SRC_DEMOTED) {
          token_rec t;
          const uint8_t* pg = slot_loc(p, row, TIER_HI, s.slot, &ip);
          get_token(pg, &p->tg[TIER_HI], ip, &t);
          demote(&t, &p->tg[TIER_LO], &lo_new[x]);
        } else {
          const uint8_t* pg = slot_loc(p, row, TIER_LO, s.slot, &ip);
          get_token(pg, &p->tg[TIER_LO], ip, &lo_new[x]);
        }
      }
      /* allocate, then free, then write */
      for (int x = 0; x < q->new_hp; x++) row[cn[2] + x] = p->list[(p->ptr[0] + aoff++) % c->n_pages];
      for (int x = 0; x < q->new_lp; x++) row[L - 1 - (cn[3] + x)] = p->list[(p->ptr[0] + aoff++) % c->n_pages];
      for (int x = 0; x < q->free_hp; x++) {
        int e = cn[2] - 1 - x;
        p->list[(p->ptr[1] + roff++) % c->n_pages] = row[e];
        row[e] = -1;
      }
      for (int x = 0; x < q->free_lp; x++) {
        int e = L - cn[3] + x;
        p->list[(p->ptr[1] + roff++) % c->n_pages] = row[e];
        row[e] = -1;
      }
      for (int x = 0; x < q->nh; x++) {
        if (!hi_dirty[x]) continue;
        int ip;
        uint8_t* pg = slot_loc(p, row, TIER_HI, x, &ip);
        put_token(pg, &p->tg[TIER_HI], ip, &hi_new[x]);
      }
      for (int x = 0; x < q->nl; x++) {
        if (!lo_dirty[x]) continue;
        int ip;
        uint8_t* pg = slot_loc(p, row, TIER_LO, x, &ip);
        put_token(pg, &p->tg[TIER_LO], ip, &lo_new[x]);
      }
      cn[0] = q->nh; cn[1] = q->nl; cn[2] = q->php; cn[3] = q->plp;
      free(hi_new); free(lo_new); free(hi_dirty); free(lo_dirty);
    }
    rs[2] = n;
  }
  p->ptr[0] += aoff;
  p->ptr[1] += roff;
  for (int hd = 0; hd < nh; hd++) { free(pl[hd].hi); free(pl[hd].lo); }
  free(pl);
  return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Decode attention — Background, attention equation, over the         */
/* dequantized mixed-precision pages (hi pages first, then lo).        */
/* ------------------------------------------------------------------ */

/* Attention of one KV head's G query heads (q: G x 128 fp16, contiguous)
 * over its stored tokens; out: G x 128 fp64; if pmax is non-NULL it
 * receives, per stored token (hi slots then lo slots), the max over the G
 * heads of its softmax probability. Returns the number of stored tokens. */
int orc_unit_attention(orc_pool* p, int layer, int slot, int kvh, const uint16_t* q, double* out,
                       double* pmax) {
  const int G = p->c.group_size;
  int32_t* cn = hcnt(p, layer, slot, kvh);
  int32_t* row = trow(p, layer, slot, kvh);
  const int n = cn[0] + cn[1];
  double* kh = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * D);
  double* vh = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * D);
  for (int j = 0; j < n; j++) {
    int tier = j < cn[0] ? TIER_HI : TIER_LO, s = j < cn[0] ? j : j - cn[0];
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
      int n = cn[0] + cn[1];
      double* pm = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
      orc_unit_attention(p, layer, slots[i], h, q + ((int64_t)i * H * G + (int64_t)h * G) * D,
                         out + ((int64_t)i * H * G + (int64_t)h * G) * D, pm);
      if (update_scores) {
        for (int j = 0; j < n; j++) {
          int tier = j < cn[0] ? TIER_HI : TIER_LO, s = j < cn[0] ? j : j - cn[0];
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
      for (int e = 0; e < p->table_len; e++) row[e] = -1;
      cn[0] = cn[1] = cn[2] = cn[3] = 0;
    }
    int32_t* rs = rstate(p, l, slot);
    rs[0] = rs[1] = rs[2] = rs[3] = 0;
  }
  return ORC_OK;
}
