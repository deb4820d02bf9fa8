/*
 * stv_oracle.c -- plain, slow, fp64 CPU oracle for one speculative tree-verify
 * round over a 3-bit quantized KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant
 * generator with the CUDA library: every definition below is written out
 * again from the method's description.
 *
 * Sources (page title, section):
 *  - "elpis" README, header table: the target keeps a 3-bit KV cache for its
 *    16 full-attention layers (12 KiB per token), 262,144-token native context.
 *  - "elpis" README, "Why fast" table: the draft's 7 nodes form an 8-row token
 *    tree, verified in one target pass; the engine commits the longest
 *    matching path plus one token; decode verify computes Q.K^T with the 3-bit
 *    K codes used as exact int8 values (int8 Q).
 *  - "elpis-lossless" README, "How" table: the 7 nodes are ranked best first;
 *    "Lossless" table: acceptance compares token ids exactly (no sampling,
 *    no thresholds).
 *  - Reddit posts (u/iamMess), second post: split-KV attention for the verify
 *    step (only the partial-result merge is implied, not its arithmetic).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - Quantizer: per (token, KV head, 32-channel group) the scale is
 *    s = fp16(max|x| / 4); the code is c = clamp(rne(x / s) + 4, 0, 7) with
 *    round-half-to-even; if s == 0 every code is 4.  Decoded value s*(c-4).
 *  - Bit layout of a block of 32 codes (three little-endian 32-bit words
 *    W0,W1,W2): for j in 0..2, k in 0..4 and m = 5j+k, code 2m sits in bits
 *    3k..3k+2 of Wj and code 2m+1 in bits 16+3k..16+3k+2 of Wj; bit b of code
 *    30 is bit 15 of Wb and bit b of code 31 is bit 31 of Wb.
 *  - Page layout per KV head (57,344 bytes, heads back to back in a page of
 *    256 tokens): K codes [256 tok][8 groups][12 B]; K scales [256 tok][8]
 *    fp16; V codes [4 tiles of 64 tok][256 ch][2 blocks of 32 tok][12 B]
 *    (channel-major: a block holds one channel's codes for 32 tokens);
 *    V scales [4 tiles][8 groups][64 tok] fp16.
 *  - Attention scale 1/sqrt(head_dim) = 1/16.  Tree rows are appended to the
 *    cache (quantized) before verify and are read back like context rows.
 *    Key j < ctx is visible to every node; key ctx+k is visible to node i iff
 *    k is an ancestor of i or i itself.
 *  - int8 Q: per (node, Q head) row, m = max|q|, qi = rne(127 q / m),
 *    sQ = fp32(m / 127); m == 0 gives qi = 0, sQ = 0.  Per 32-channel group
 *    the integer dot I_g = sum qi * (c - 4); S = sQ * sum_g sK_g * I_g / 16.
 *  - Acceptance: edge p->c matches iff draft[c] == argmax[p].  Among paths
 *    from the root whose every edge matches, take the longest; among equally
 *    long ones, the lexicographically smallest sequence of node indices
 *    (lower index = better ranked draft).  n_commit = path length (accepted
 *    depth + 1); out_ids = drafts of path[1..], then argmax[path[last]].
 *  - Commit: slot ctx+i takes the packed row of slot ctx+path[i], i < n_commit.
 *
 * All floating point is fp64 (IEEE, default round-to-nearest-even); softmax
 * is two-pass (max, then sum), with no online rescaling and no blocking.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define HEAD_DIM 256
#define GROUP 32
#define N_GROUPS (HEAD_DIM / GROUP)
#define PAGE_TOK 256
#define TILE_TOK 64

/* Byte offsets inside one KV head's 57,344-byte block of a page. */
#define OFF_K_CODES 0
#define OFF_K_SCALES (PAGE_TOK * N_GROUPS * 12)               /* 24576 */
#define OFF_V_CODES (OFF_K_SCALES + PAGE_TOK * N_GROUPS * 2)  /* 28672 */
#define OFF_V_SCALES (OFF_V_CODES + PAGE_TOK * N_GROUPS * 12) /* 53248 */
#define HEAD_BYTES (OFF_V_SCALES + PAGE_TOK * N_GROUPS * 2)   /* 57344 */

enum {
  ORC_OK = 0,
  ORC_BAD_ARG = -1,
  ORC_BAD_TREE = -2,
  ORC_BAD_PAGE = -3,
};

int orc_head_bytes(void) { return HEAD_BYTES; }



/* ------------------------------------------------------------------------ */
/* IEEE binary16 <-> binary64.                                              */
/* ------------------------------------------------------------------------ */

double orc_half_to_double(uint16_t h) {
  int sign = h >> 15, e = (h >> 10) & 31, man = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)man, -24);
  else if (e == 31)
    v = man ? NAN : INFINITY;
  else
    v = ldexp((double)(man + 1024), e - 25);
  return sign ? -v : v;
}

/* Round to the nearest binary16, ties to even. */
uint16_t orc_double_to_half(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isnan(x)) return 0x7e00;
  if (a < ldexp(1.0, -14)) {
    /* subnormal range: the quantum is 2^-24; 1024 quanta is the smallest
     * normal, whose encoding is also 1024. */
    double r = rint(a * 16777216.0);
    return sign | (uint16_t)r;
  }
  int e;
  frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
  double r = rint(ldexp(a, 11 - e)); /* 11 significant bits */
  int E = e - 1;
  if (r == 2048.0) {
    r = 1024.0;
    E += 1;
  }
  if (E > 15) return sign | 0x7c00;
  return sign | (uint16_t)((E + 15) << 10) | (uint16_t)((int)r - 1024);
}

float orc_double_to_float(double x) { return (float)x; }

/* ------------------------------------------------------------------------
 * Second cache format (next row f3): int4 with one scale per token and KV
 * head ("elpis" README mirror, syv-ai README, int4 KV section: the stock
 * int4_per_token_head cache).  Reading (the pages give no formula): per
 * (token, KV head) m = max|x| over its 256 values, s = fp16(m / 7),
 * c = clamp(rne(x / s), -8, 7) (all 0 when s == 0), stored as u = c + 8 in 4
 * bits; decoded value s * c.  Layout per KV head (66,560 bytes): K codes
 * [256 tok][32 words], K scales [256] fp16, V codes [4 tiles of 64 tok]
 * [256 ch][8 words] (channel-major: a word holds one channel's codes for 8
 * tokens), V scales [256] fp16.  Inside a word of 8 elements e0..e7,
 * element e sits at bit 4*(e/2) (even e) or 16 + 4*(e/2) (odd e).
 * The format of a pool follows from its page stride: hkv * 57,344 bytes for
 * the 3-bit cache, hkv * 66,560 for this one.
 */
#define I4_OFF_K_CODES 0
#define I4_OFF_K_SCALES (PAGE_TOK * 128)                /* 32768 */
#define I4_OFF_V_CODES (I4_OFF_K_SCALES + PAGE_TOK * 2)  /* 33280 */
#define I4_OFF_V_SCALES (I4_OFF_V_CODES + PAGE_TOK * 128) /* 66048 */
#define I4_HEAD_BYTES (I4_OFF_V_SCALES + PAGE_TOK * 2)   /* 66560 */

int orc_head_bytes_i4(void) { return I4_HEAD_BYTES; }

/* Bit position of element e (0..7) inside its word. */
static int i4_pos(int e) { return ((e & 1) ? 16 : 0) + 4 * (e >> 1); }

/* Quantize one token-head row of 256 fp16 values: scale and codes u = c + 8. */
void orc_quantize_row_i4(const uint16_t* x, uint16_t* s_out, uint8_t* u) {
  double m = 0.0;
  for (int i = 0; i < HEAD_DIM; ++i) {
    double a = fabs(orc_half_to_double(x[i]));
    if (a > m) m = a;
  }
  uint16_t s = orc_double_to_half(m / 7.0);
  double sd = orc_half_to_double(s);
  for (int i = 0; i < HEAD_DIM; ++i) {
    double c = sd == 0.0 ? 0.0 : rint(orc_half_to_double(x[i]) / sd);
    if (c < -8.0) c = -8.0;
    if (c > 7.0) c = 7.0;
    u[i] = (uint8_t)(c + 8.0);
  }
  *s_out = s;
}

/* ------------------------------------------------------------------------
 * Third cache format (next row f3): the KVarN-style 4/2-bit cache (Reddit
 * posts (u/iamMess), "Now added" list: a KVarN 4/2-bit KV cache; syv-ai
 * README (mirror), DFlash2 at 240k: CTX=huge uses it).  The pages name it
 * and give its cost, not its quantizer.  Reading: the 3-bit cache's
 * quantizer at other widths, 4 bits for K and 2 bits for V, one fp16 scale
 * per (token, KV head, group of 32 channels): for b bits, h = 2^(b-1),
 * s = fp16(m / h), c = clamp(rne(x / s), -h, h - 1) (all 0 when s == 0),
 * stored as u = c + h; decoded value s * c.  (At b = 3 this is the 3-bit
 * cache's quantizer, whose code is u.)  Layout per KV head (57,344 bytes,
 * the 3-bit cache's size: 4 + 2 bits against 3 + 3):
 *   [0, 32768)      K codes  [256 tok][8 groups][4 words]; a word holds 8
 *                   channels, element e at bit 4*(e/2) + 16*(e%2)
 *   [32768, 36864)  K scales [256 tok][8 groups] fp16
 *   [36864, 53248)  V codes  [4 tiles of 64 tok][256 ch][4 words]; a word
 *                   holds one channel's codes for 16 tokens, token t at
 *                   bit 2*(t/2) + 16*(t%2)
 *   [53248, 57344)  V scales [4 tiles][8 groups][64 tok] fp16 (as in the
 *                   3-bit cache)
 * Its page stride equals the 3-bit cache's, so callers name the format.
 */
#define KV2_OFF_K_CODES 0
#define KV2_OFF_K_SCALES (PAGE_TOK * N_GROUPS * 16)                  /* 32768 */
#define KV2_OFF_V_CODES (KV2_OFF_K_SCALES + PAGE_TOK * N_GROUPS * 2)  /* 36864 */
#define KV2_OFF_V_SCALES (KV2_OFF_V_CODES + PAGE_TOK * HEAD_DIM / 4)  /* 53248 */
#define KV2_HEAD_BYTES (KV2_OFF_V_SCALES + PAGE_TOK * N_GROUPS * 2)   /* 57344 */

/* Bit position of token t (0..15) inside a 2-bit V word. */
static int v2_pos(int t) { return ((t & 1) ? 16 : 0) + 2 * (t >> 1); }

/* Quantize 32 fp16 values at b bits: one fp16 scale and codes u = c + h. */
void orc_quantize_group_bits(const uint16_t* x, int bits, uint16_t* s_out, uint8_t* u) {
  const double h = (double)(1 << (bits - 1));
  double m = 0.0;
  for (int i = 0; i < GROUP; ++i) {
    double a = fabs(orc_half_to_double(x[i]));
    if (a > m) m = a;
  }
  uint16_t s = orc_double_to_half(m / h);
  double sd = orc_half_to_double(s);
  for (int i = 0; i < GROUP; ++i) {
    double c = sd == 0.0 ? 0.0 : rint(orc_half_to_double(x[i]) / sd);
    if (c < -h) c = -h;
    if (c > h - 1.0) c = h - 1.0;
    u[i] = (uint8_t)(c + h);
  }
  *s_out = s;
}

/* ------------------------------------------------------------------------ */
/* 3-bit group quantizer and the block bit layout.                          */
/* ------------------------------------------------------------------------ */

/* Quantize 32 fp16 values: one fp16 scale, 32 codes in 0..7. */
void orc_quantize_group(const uint16_t* x, uint16_t* s_out, uint8_t* codes) {
  double m = 0.0;
  for (int i = 0; i < GROUP; ++i) {
    double a = fabs(orc_half_to_double(x[i]));
    if (a > m) m = a;
  }
  uint16_t s = orc_double_to_half(m / 4.0);
  double sd = orc_half_to_double(s);
  for (int i = 0; i < GROUP; ++i) {
    if (sd == 0.0) {
      codes[i] = 4;
      continue;
    }
    double c = rint(orc_half_to_double(x[i]) / sd) + 4.0;
    if (c < 0.0) c = 0.0;
    if (c > 7.0) c = 7.0;
    codes[i] = (uint8_t)c;
  }
  *s_out = s;
}

/* Where bit b of code i of a 32-code block lives. */
static void bit_place(int i, int b, int* word, int* bit) {
  if (i < 30) {
    int m = i >> 1;
    *word = m / 5;
    *bit = ((i & 1) ? 16 : 0) + 3 * (m % 5) + b;
  } else {
    *word = b;
    *bit = (i == 30) ? 15 : 31;
  }
}

void orc_pack_block(const uint8_t* codes, uint32_t* w) {
  w[0] = w[1] = w[2] = 0;
  for (int i = 0; i < GROUP; ++i)
    for (int b = 0; b < 3; ++b)
      if ((codes[i] >> b) & 1) {
        int wd, bt;
        bit_place(i, b, &wd, &bt);
        w[wd] |= 1u << bt;
      }
}

uint8_t orc_block_code(const uint32_t* w, int i) {
  uint8_t c = 0;
  for (int b = 0; b < 3; ++b) {
    int wd, bt;
    bit_place(i, b, &wd, &bt);
    c |= (uint8_t)(((w[wd] >> bt) & 1u) << b);
  }
  return c;
}

static void block_set_code(uint32_t* w, int i, uint8_t c) {
  for (int b = 0; b < 3; ++b) {
    int wd, bt;
    bit_place(i, b, &wd, &bt);
    w[wd] &= ~(1u << bt);
    w[wd] |= (uint32_t)((c >> b) & 1) << bt;
  }
}

/* ------------------------------------------------------------------------ */
/* Paged cache addressing.                                                  */
/* ------------------------------------------------------------------------ */

typedef struct {
  uint8_t* pool;
  int64_t page_bytes;
  int32_t pool_pages;
  int32_t hkv;
  const int32_t* page_tables; /* all sequences' tables, concatenated */
  const int32_t* pt_offsets;  /* [n_seqs + 1] */
  int fmt;                    /* 0: 3-bit groups of 32, 1: int4 per token and head, 2: K 4 bits / V 2 bits */
  int64_t head_bytes;
} cache_view;

/* Set the pool's format; ORC_BAD_ARG if the page stride does not match it. */
static int view_format(cache_view* cv, int fmt) {
  static const int64_t head[3] = {HEAD_BYTES, I4_HEAD_BYTES, KV2_HEAD_BYTES};
  if (fmt < 0 || fmt > 2 || cv->page_bytes != (int64_t)cv->hkv * head[fmt]) return ORC_BAD_ARG;
  cv->fmt = fmt;
  cv->head_bytes = head[fmt];
  return ORC_OK;
}

/* Base of KV head h's block for token `tok` of sequence `seq`, or NULL. */
static uint8_t* head_block(const cache_view* cv, int seq, int64_t tok, int h) {
  int64_t lp = tok / PAGE_TOK;
  int64_t np = cv->pt_offsets[seq + 1] - cv->pt_offsets[seq];
  if (tok < 0 || lp >= np) return NULL;
  int32_t page = cv->page_tables[cv->pt_offsets[seq] + lp];
  if (page < 0 || page >= cv->pool_pages) return NULL;
  return cv->pool + (int64_t)page * cv->page_bytes + (int64_t)h * cv->head_bytes;
}

static void load_words(const uint8_t* p, uint32_t* w) { memcpy(w, p, 12); }
static void store_words(uint8_t* p, const uint32_t* w) { memcpy(p, w, 12); }

static uint16_t load_u16(const uint8_t* p) {
  uint16_t v;
  memcpy(&v, p, 2);
  return v;
}
static void store_u16(uint8_t* p, uint16_t v) { memcpy(p, &v, 2); }

/* K: codes and scale of (slot, group). */
static uint8_t* k_words(uint8_t* hb, int slot, int g) { return hb + OFF_K_CODES + slot * 96 + g * 12; }
static uint8_t* k_scale(uint8_t* hb, int slot, int g) { return hb + OFF_K_SCALES + slot * 16 + g * 2; }
/* V: channel-major block of 32 tokens holding `slot`; position slot % 32. */
static uint8_t* v_words(uint8_t* hb, int slot, int ch) {
  return hb + OFF_V_CODES + (slot / TILE_TOK) * (HEAD_DIM * 24) + ch * 24 + ((slot % TILE_TOK) / 32) * 12;
}
static uint8_t* v_scale(uint8_t* hb, int slot, int g) {
  return hb + OFF_V_SCALES + (slot / TILE_TOK) * (N_GROUPS * TILE_TOK * 2) + g * (TILE_TOK * 2) + (slot % TILE_TOK) * 2;
}

/* Decode K (which = 0) or V (which = 1) of one token and head: 256 values. */
/* int4 cache: code u of element `ch` (K) or `slot` (V) of one token and head. */
static int i4_code(uint8_t* hb, int which, int slot, int ch) {
  uint32_t w;
  if (which == 0) {
    memcpy(&w, hb + I4_OFF_K_CODES + slot * 128 + (ch / 8) * 4, 4);
    return (int)((w >> i4_pos(ch % 8)) & 15u);
  }
  int within = slot % TILE_TOK;
  memcpy(&w, hb + I4_OFF_V_CODES + (slot / TILE_TOK) * (HEAD_DIM * 32) + ch * 32 + (within / 8) * 4, 4);
  return (int)((w >> i4_pos(within % 8)) & 15u);
}
static uint8_t* i4_scale(uint8_t* hb, int which, int slot) {
  return hb + (which == 0 ? I4_OFF_K_SCALES : I4_OFF_V_SCALES) + slot * 2;
}

/* K 4 / V 2-bit cache: code u of channel `ch` of one token and head. */
static uint8_t* kv2_k_word(uint8_t* hb, int slot, int ch) {
  return hb + KV2_OFF_K_CODES + slot * 128 + (ch / GROUP) * 16 + ((ch % GROUP) / 8) * 4;
}
static uint8_t* kv2_v_word(uint8_t* hb, int slot, int ch) {
  int within = slot % TILE_TOK;
  return hb + KV2_OFF_V_CODES + (slot / TILE_TOK) * (HEAD_DIM * 16) + ch * 16 + (within / 16) * 4;
}
static int kv2_code(uint8_t* hb, int which, int slot, int ch) {
  uint32_t w;
  if (which == 0) {
    memcpy(&w, kv2_k_word(hb, slot, ch), 4);
    return (int)((w >> i4_pos(ch % 8)) & 15u);
  }
  memcpy(&w, kv2_v_word(hb, slot, ch), 4);
  return (int)((w >> v2_pos(slot % 16)) & 3u);
}
static uint8_t* kv2_k_scale(uint8_t* hb, int slot, int g) { return hb + KV2_OFF_K_SCALES + slot * 16 + g * 2; }

static int decode_row(const cache_view* cv, int seq, int64_t tok, int h, int which, double* out) {
  uint8_t* hb = head_block(cv, seq, tok, h);
  if (!hb) return ORC_BAD_PAGE;
  int slot = (int)(tok % PAGE_TOK);
  if (cv->fmt == 2) {
    for (int g = 0; g < N_GROUPS; ++g) {
      double s = orc_half_to_double(load_u16(which == 0 ? kv2_k_scale(hb, slot, g) : v_scale(hb, slot, g)));
      for (int i = 0; i < GROUP; ++i)
        out[g * GROUP + i] = s * (kv2_code(hb, which, slot, g * GROUP + i) - (which == 0 ? 8 : 2));
    }
    return ORC_OK;
  }
  if (cv->fmt == 1) {
    double s = orc_half_to_double(load_u16(i4_scale(hb, which, slot)));
    for (int c = 0; c < HEAD_DIM; ++c) out[c] = s * (i4_code(hb, which, slot, c) - 8);
    return ORC_OK;
  }
  for (int g = 0; g < N_GROUPS; ++g) {
    if (which == 0) {
      uint32_t w[3];
      load_words(k_words(hb, slot, g), w);
      double s = orc_half_to_double(load_u16(k_scale(hb, slot, g)));
      for (int i = 0; i < GROUP; ++i) out[g * GROUP + i] = s * ((int)orc_block_code(w, i) - 4);
    } else {
      double s = orc_half_to_double(load_u16(v_scale(hb, slot, g)));
      for (int i = 0; i < GROUP; ++i) {
        uint32_t w[3];
        load_words(v_words(hb, slot, g * GROUP + i), w);
        out[g * GROUP + i] = s * ((int)orc_block_code(w, slot % 32) - 4);
      }
    }
  }
  return ORC_OK;
}

/* K's integer values (code - 4 for the 3-bit cache, u - 8 for int4 and for
 * the 4-bit K of the K 4 / V 2-bit cache) and
 * per-group scales of one token and head, for the int8 definition (the
 * int4 cache has one scale per token: every group gets it). */
static int k_codes_row(const cache_view* cv, int seq, int64_t tok, int h, int8_t* kv, double* scales) {
  uint8_t* hb = head_block(cv, seq, tok, h);
  if (!hb) return ORC_BAD_PAGE;
  int slot = (int)(tok % PAGE_TOK);
  if (cv->fmt == 2) {
    for (int g = 0; g < N_GROUPS; ++g) scales[g] = orc_half_to_double(load_u16(kv2_k_scale(hb, slot, g)));
    for (int c = 0; c < HEAD_DIM; ++c) kv[c] = (int8_t)(kv2_code(hb, 0, slot, c) - 8);
    return ORC_OK;
  }
  if (cv->fmt == 1) {
    double s = orc_half_to_double(load_u16(i4_scale(hb, 0, slot)));
    for (int g = 0; g < N_GROUPS; ++g) scales[g] = s;
    for (int c = 0; c < HEAD_DIM; ++c) kv[c] = (int8_t)(i4_code(hb, 0, slot, c) - 8);
    return ORC_OK;
  }
  for (int g = 0; g < N_GROUPS; ++g) {
    uint32_t w[3];
    load_words(k_words(hb, slot, g), w);
    scales[g] = orc_half_to_double(load_u16(k_scale(hb, slot, g)));
    for (int i = 0; i < GROUP; ++i) kv[g * GROUP + i] = (int8_t)((int)orc_block_code(w, i) - 4);
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* kv_append_pack: quantize fp16 K/V rows into the paged 3-bit cache.       */
/* ------------------------------------------------------------------------ */

int orc_kv_append(uint8_t* pool, int64_t page_bytes, int32_t pool_pages, int32_t hkv,
                  const int32_t* page_tables, const int32_t* pt_offsets, int n_seqs,
                  const uint16_t* k, const uint16_t* v, /* [n_rows][hkv][256] */
                  const int32_t* row_seq, const int32_t* row_pos, int n_rows, int fmt) {
  cache_view cv = {pool, page_bytes, pool_pages, hkv, page_tables, pt_offsets};
  if (view_format(&cv, fmt) != ORC_OK) return ORC_BAD_ARG;
  for (int r = 0; r < n_rows; ++r) {
    int seq = row_seq[r];
    if (seq < 0 || seq >= n_seqs) return ORC_BAD_ARG;
    for (int h = 0; h < hkv; ++h) {
      uint8_t* hb = head_block(&cv, seq, row_pos[r], h);
      if (!hb) return ORC_BAD_PAGE;
      int slot = row_pos[r] % PAGE_TOK;
      const uint16_t* kr = k + ((int64_t)r * hkv + h) * HEAD_DIM;
      const uint16_t* vr = v + ((int64_t)r * hkv + h) * HEAD_DIM;
      if (cv.fmt == 2) { /* K 4 bits, V 2 bits, per group of 32 channels */
        for (int g = 0; g < N_GROUPS; ++g) {
          uint16_t s;
          uint8_t u[GROUP];
          orc_quantize_group_bits(kr + g * GROUP, 4, &s, u);
          for (int wd = 0; wd < 4; ++wd) {
            uint32_t w = 0;
            for (int e = 0; e < 8; ++e) w |= (uint32_t)u[8 * wd + e] << i4_pos(e);
            memcpy(kv2_k_word(hb, slot, g * GROUP + 8 * wd), &w, 4);
          }
          store_u16(kv2_k_scale(hb, slot, g), s);
          orc_quantize_group_bits(vr + g * GROUP, 2, &s, u);
          store_u16(v_scale(hb, slot, g), s);
          for (int i = 0; i < GROUP; ++i) {
            uint8_t* p = kv2_v_word(hb, slot, g * GROUP + i);
            uint32_t w;
            memcpy(&w, p, 4);
            w = (w & ~(3u << v2_pos(slot % 16))) | ((uint32_t)u[i] << v2_pos(slot % 16));
            memcpy(p, &w, 4);
          }
        }
        continue;
      }
      if (cv.fmt == 1) { /* int4 per token and head */
        uint16_t s;
        uint8_t u[HEAD_DIM];
        orc_quantize_row_i4(kr, &s, u);
        for (int wd = 0; wd < HEAD_DIM / 8; ++wd) {
          uint32_t w = 0;
          for (int e = 0; e < 8; ++e) w |= (uint32_t)u[8 * wd + e] << i4_pos(e);
          memcpy(hb + I4_OFF_K_CODES + slot * 128 + wd * 4, &w, 4);
        }
        store_u16(i4_scale(hb, 0, slot), s);
        orc_quantize_row_i4(vr, &s, u);
        store_u16(i4_scale(hb, 1, slot), s);
        int within = slot % TILE_TOK;
        for (int c = 0; c < HEAD_DIM; ++c) {
          uint8_t* p = hb + I4_OFF_V_CODES + (slot / TILE_TOK) * (HEAD_DIM * 32) + c * 32 + (within / 8) * 4;
          uint32_t w;
          memcpy(&w, p, 4);
          w = (w & ~(15u << i4_pos(within % 8))) | ((uint32_t)u[c] << i4_pos(within % 8));
          memcpy(p, &w, 4);
        }
        continue;
      }
      for (int g = 0; g < N_GROUPS; ++g) {
        uint16_t s;
        uint8_t codes[GROUP];
        uint32_t w[3];
        /* K: one token's group of 32 channels is one block. */
        orc_quantize_group(kr + g * GROUP, &s, codes);
        orc_pack_block(codes, w);
        store_words(k_words(hb, slot, g), w);
        store_u16(k_scale(hb, slot, g), s);
        /* V: same quantizer; each channel's code goes to that channel's
         * block of 32 tokens. */
        orc_quantize_group(vr + g * GROUP, &s, codes);
        store_u16(v_scale(hb, slot, g), s);
        for (int i = 0; i < GROUP; ++i) {
          uint8_t* p = v_words(hb, slot, g * GROUP + i);
          load_words(p, w);
          block_set_code(w, slot % 32, codes[i]);
          store_words(p, w);
        }
      }
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Tree: ancestor-or-self sets.                                             */
/* ------------------------------------------------------------------------ */

/* parent[0] == -1 and 0 <= parent[i] < i for i >= 1. */
int orc_check_tree(const int32_t* parent, int t) {
  if (t < 1 || t > 32) return ORC_BAD_TREE;
  if (parent[0] != -1) return ORC_BAD_TREE;
  for (int i = 1; i < t; ++i)
    if (parent[i] < 0 || parent[i] >= i) return ORC_BAD_TREE;
  return ORC_OK;
}

/* anc[i] bit k set iff node k is node i or one of its ancestors. */
int orc_ancestors(const int32_t* parent, int t, uint32_t* anc) {
  if (orc_check_tree(parent, t) != ORC_OK) return ORC_BAD_TREE;
  for (int i = 0; i < t; ++i) {
    uint32_t m = 0;
    for (int n = i; n >= 0; n = parent[n]) m |= 1u << n;
    anc[i] = m;
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* int8 Q quantizer.                                                        */
/* ------------------------------------------------------------------------ */

void orc_quantize_q_int8(const uint16_t* q, int8_t* qi, float* sq) {
  double m = 0.0;
  for (int c = 0; c < HEAD_DIM; ++c) {
    double a = fabs(orc_half_to_double(q[c]));
    if (a > m) m = a;
  }
  for (int c = 0; c < HEAD_DIM; ++c)
    qi[c] = (m == 0.0) ? 0 : (int8_t)rint(127.0 * orc_half_to_double(q[c]) / m);
  *sq = (float)(m / 127.0);
}

/* Integer per-group dots I_g = sum_{c in g} qi_c * (code_c - 4). */
static void int8_group_dots(const int8_t* qi, const int8_t* kv, int64_t* dots) {
  for (int g = 0; g < N_GROUPS; ++g) {
    int64_t acc = 0;
    for (int i = 0; i < GROUP; ++i) acc += (int64_t)qi[g * GROUP + i] * (int64_t)kv[g * GROUP + i];
    dots[g] = acc;
  }
}

/* ------------------------------------------------------------------------ */
/* Tree-masked attention over the cache (exact and int8 definitions).       */
/* ------------------------------------------------------------------------ */

typedef struct {
  const cache_view* cv;
  const int32_t* ctx;
  const uint16_t* q;
  const int32_t* parent;
  int t, hq, hkv, path;
  const int32_t* rows; /* [n][3]: seq, node, q head */
  double* out;
  int n_rows;
  int next; /* next row to take */
  pthread_mutex_t lock;
  int err;
} attn_job;

static int attention_row(attn_job* jb, int r) {
  const cache_view* cv = jb->cv;
  int seq = jb->rows[3 * r], node = jb->rows[3 * r + 1], qh = jb->rows[3 * r + 2];
  int t = jb->t, hq = jb->hq, G = hq / jb->hkv, h = qh / G;
  if (node < 0 || node >= t || qh < 0 || qh >= hq) return ORC_BAD_ARG;
  uint32_t anc[32];
  if (orc_ancestors(jb->parent + (int64_t)seq * t, t, anc) != ORC_OK) return ORC_BAD_TREE;
  int64_t ctx = jb->ctx[seq];
  const uint16_t* qrow = jb->q + (((int64_t)seq * t + node) * hq + qh) * HEAD_DIM;

  double qd[HEAD_DIM];
  for (int c = 0; c < HEAD_DIM; ++c) qd[c] = orc_half_to_double(qrow[c]);
  int8_t qi[HEAD_DIM];
  float sq = 0.f;
  if (jb->path == 1) orc_quantize_q_int8(qrow, qi, &sq);

  /* Visible keys: the whole context, then the node's ancestors-or-self. */
  int64_t n_vis = ctx;
  for (int k = 0; k < t; ++k)
    if ((anc[node] >> k) & 1) ++n_vis;
  int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * n_vis);
  double* score = (double*)malloc(sizeof(double) * n_vis);
  if (!keys || !score) {
    free(keys);
    free(score);
    return ORC_BAD_ARG;
  }
  int64_t n = 0;
  for (int64_t j = 0; j < ctx; ++j) keys[n++] = j;
  for (int k = 0; k < t; ++k)
    if ((anc[node] >> k) & 1) keys[n++] = ctx + k;

  /* Pass 1: scores S_j = q . k_j / 16 and their maximum. */
  double smax = -INFINITY;
  int rc = ORC_OK;
  for (int64_t a = 0; a < n_vis && rc == ORC_OK; ++a) {
    double s = 0.0;
    if (jb->path == 0) {
      double kd[HEAD_DIM];
      rc = decode_row(cv, seq, keys[a], h, 0, kd);
      for (int c = 0; c < HEAD_DIM; ++c) s += qd[c] * kd[c];
      s /= 16.0;
    } else {
      int8_t kv[HEAD_DIM];
      double sk[N_GROUPS];
      int64_t dots[N_GROUPS];
      rc = k_codes_row(cv, seq, keys[a], h, kv, sk);
      int8_group_dots(qi, kv, dots);
      for (int g = 0; g < N_GROUPS; ++g) s += sk[g] * (double)dots[g];
      s = (double)sq * s / 16.0;
    }
    score[a] = s;
    if (s > smax) smax = s;
  }
  /* Pass 2: softmax weights and the weighted sum of decoded V rows. */
  double l = 0.0, o[HEAD_DIM];
  for (int c = 0; c < HEAD_DIM; ++c) o[c] = 0.0;
  for (int64_t a = 0; a < n_vis && rc == ORC_OK; ++a) {
    double p = exp(score[a] - smax);
    double vd[HEAD_DIM];
    rc = decode_row(cv, seq, keys[a], h, 1, vd);
    l += p;
    for (int c = 0; c < HEAD_DIM; ++c) o[c] += p * vd[c];
  }
  double* dst = jb->out + (int64_t)r * HEAD_DIM;
  for (int c = 0; c < HEAD_DIM; ++c) dst[c] = o[c] / l;
  free(keys);
  free(score);
  return rc;
}

static void* attn_worker(void* arg) {
  attn_job* jb = (attn_job*)arg;
  for (;;) {
    pthread_mutex_lock(&jb->lock);
    int r = jb->next++;
    pthread_mutex_unlock(&jb->lock);
    if (r >= jb->n_rows) break;
    int rc = attention_row(jb, r);
    if (rc != ORC_OK) {
      pthread_mutex_lock(&jb->lock);
      jb->err = rc;
      pthread_mutex_unlock(&jb->lock);
    }
  }
  return NULL;
}

/*
 * Attention output (fp64) of the listed (seq, node, q head) rows.
 * path 0 = exact definition (fp16 Q times decoded K), 1 = int8 definition.
 * q: [n_seqs][t][hq][256] fp16 bits; parent: [n_seqs][t]; ctx: [n_seqs].
 */
int orc_attention(const uint8_t* pool, int64_t page_bytes, int32_t pool_pages, int32_t hq, int32_t hkv,
                  const int32_t* page_tables, const int32_t* pt_offsets, const int32_t* ctx, int n_seqs,
                  const uint16_t* q, const int32_t* parent, int t, int path, const int32_t* rows, int n_rows,
                  double* out, int n_threads, int fmt) {
  if (hkv < 1 || hq % hkv != 0 || t < 1 || t > 32 || (path != 0 && path != 1)) return ORC_BAD_ARG;
  for (int r = 0; r < n_rows; ++r)
    if (rows[3 * r] < 0 || rows[3 * r] >= n_seqs) return ORC_BAD_ARG;
  cache_view cv = {(uint8_t*)pool, page_bytes, pool_pages, hkv, page_tables, pt_offsets};
  if (view_format(&cv, fmt) != ORC_OK) return ORC_BAD_ARG;
  attn_job jb;
  jb.cv = &cv;
  jb.ctx = ctx;
  jb.q = q;
  jb.parent = parent;
  jb.t = t;
  jb.hq = hq;
  jb.hkv = hkv;
  jb.path = path;
  jb.rows = rows;
  jb.out = out;
  jb.n_rows = n_rows;
  jb.next = 0;
  jb.err = ORC_OK;
  pthread_mutex_init(&jb.lock, NULL);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  pthread_t th[256];
  int started = 0;
  for (int i = 1; i < n_threads; ++i)
    if (pthread_create(&th[started], NULL, attn_worker, &jb) == 0) ++started;
  attn_worker(&jb);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&jb.lock);
  return jb.err;
}

/* The int8 path's integer dots I_g for keys [tok_begin, tok_end) of one row.
 * out: [tok_end - tok_begin][8] int32 (|I_g| <= 32*127*4 fits easily). */
int orc_int8_dots(const uint8_t* pool, int64_t page_bytes, int32_t pool_pages, int32_t hq, int32_t hkv,
                  const int32_t* page_tables, const int32_t* pt_offsets, int seq, const uint16_t* qrow,
                  int qhead, int64_t tok_begin, int64_t tok_end, int32_t* out, int fmt) {
  cache_view cv = {(uint8_t*)pool, page_bytes, pool_pages, hkv, page_tables, pt_offsets};
  if (view_format(&cv, fmt) != ORC_OK) return ORC_BAD_ARG;
  int h = qhead / (hq / hkv);
  int8_t qi[HEAD_DIM];
  float sq;
  orc_quantize_q_int8(qrow, qi, &sq);
  for (int64_t j = tok_begin; j < tok_end; ++j) {
    int8_t kv[HEAD_DIM];
    double sk[N_GROUPS];
    int64_t dots[N_GROUPS];
    if (k_codes_row(&cv, seq, j, h, kv, sk) != ORC_OK) return ORC_BAD_PAGE;
    int8_group_dots(qi, kv, dots);
    for (int g = 0; g < N_GROUPS; ++g) out[(j - tok_begin) * N_GROUPS + g] = (int32_t)dots[g];
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Greedy tree acceptance.                                                  */
/* ------------------------------------------------------------------------ */

/* Root-first node sequence ending at `node`; returns its length. */
static int root_path(const int32_t* parent, int node, int32_t* seq_out) {
  int32_t rev[32];
  int n = 0;
  for (int x = node; x >= 0; x = parent[x]) rev[n++] = x;
  for (int i = 0; i < n; ++i) seq_out[i] = rev[n - 1 - i];
  return n;
}

int orc_tree_accept(const int32_t* parent, const int32_t* draft, const int32_t* argmax, int t, int32_t* n_commit,
                    int32_t* path, int32_t* out_ids) {
  if (orc_check_tree(parent, t) != ORC_OK) return ORC_BAD_TREE;
  /* ok[i]: every edge from the root to i matches (nodes in index order, so
   * a parent is settled before its children). */
  int ok[32], depth[32];
  ok[0] = 1;
  depth[0] = 0;
  for (int i = 1; i < t; ++i) {
    ok[i] = ok[parent[i]] && draft[i] == argmax[parent[i]];
    depth[i] = depth[parent[i]] + 1;
  }
  int best = 0;
  int32_t best_path[32], cand[32];
  int best_len = root_path(parent, 0, best_path);
  for (int i = 1; i < t; ++i) {
    if (!ok[i]) continue;
    int len = root_path(parent, i, cand);
    int better = len > best_len;
    if (len == best_len) {
      for (int a = 0; a < len; ++a)
        if (cand[a] != best_path[a]) {
          better = cand[a] < best_path[a];
          break;
        }
    }
    if (better) {
      best = i;
      best_len = len;
      memcpy(best_path, cand, sizeof(int32_t) * len);
    }
  }
  (void)depth;
  *n_commit = best_len;
  for (int a = 0; a < best_len; ++a) path[a] = best_path[a];
  for (int a = 1; a < best_len; ++a) out_ids[a - 1] = draft[best_path[a]];
  out_ids[best_len - 1] = argmax[best];
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* kv_commit: compact the accepted rows to slots ctx .. ctx+n_commit-1.      */
/* ------------------------------------------------------------------------ */

int orc_kv_commit(uint8_t* pool, int64_t page_bytes, int32_t pool_pages, int32_t hkv, const int32_t* page_tables,
                  const int32_t* pt_offsets, const int32_t* ctx, int n_seqs, const int32_t* n_commit,
                  const int32_t* path, int t, int fmt) {
  cache_view cv = {pool, page_bytes, pool_pages, hkv, page_tables, pt_offsets};
  if (view_format(&cv, fmt) != ORC_OK) return ORC_BAD_ARG;
  for (int s = 0; s < n_seqs; ++s) {
    int n = n_commit[s];
    if (n < 1 || n > t) return ORC_BAD_ARG;
    for (int h = 0; h < hkv; ++h) {
      if (cv.fmt == 2) { /* K 4 / V 2: K codes and both scale rows move whole; V codes channel by channel */
        uint8_t kc2[32][128], ks2[32][16], vs2[32][16], vu2[32][HEAD_DIM];
        for (int i = 0; i < n; ++i) {
          int64_t src = (int64_t)ctx[s] + path[(int64_t)s * t + i];
          uint8_t* hb = head_block(&cv, s, src, h);
          if (!hb) return ORC_BAD_PAGE;
          int slot = (int)(src % PAGE_TOK);
          memcpy(kc2[i], hb + KV2_OFF_K_CODES + slot * 128, 128);
          memcpy(ks2[i], kv2_k_scale(hb, slot, 0), 16);
          for (int g = 0; g < N_GROUPS; ++g) memcpy(vs2[i] + 2 * g, v_scale(hb, slot, g), 2);
          for (int c = 0; c < HEAD_DIM; ++c) vu2[i][c] = (uint8_t)kv2_code(hb, 1, slot, c);
        }
        for (int i = 0; i < n; ++i) {
          int64_t dst = (int64_t)ctx[s] + i;
          uint8_t* hb = head_block(&cv, s, dst, h);
          if (!hb) return ORC_BAD_PAGE;
          int slot = (int)(dst % PAGE_TOK);
          memcpy(hb + KV2_OFF_K_CODES + slot * 128, kc2[i], 128);
          memcpy(kv2_k_scale(hb, slot, 0), ks2[i], 16);
          for (int g = 0; g < N_GROUPS; ++g) memcpy(v_scale(hb, slot, g), vs2[i] + 2 * g, 2);
          for (int c = 0; c < HEAD_DIM; ++c) {
            uint8_t* p = kv2_v_word(hb, slot, c);
            uint32_t w;
            memcpy(&w, p, 4);
            w = (w & ~(3u << v2_pos(slot % 16))) | ((uint32_t)vu2[i][c] << v2_pos(slot % 16));
            memcpy(p, &w, 4);
          }
        }
        continue;
      }
      if (cv.fmt == 1) { /* int4: K codes and both scales move whole; V nibbles channel by channel */
        uint8_t kc4[32][128], sc4[32][4], vu[32][HEAD_DIM];
        for (int i = 0; i < n; ++i) {
          int64_t src = (int64_t)ctx[s] + path[(int64_t)s * t + i];
          uint8_t* hb = head_block(&cv, s, src, h);
          if (!hb) return ORC_BAD_PAGE;
          int slot = (int)(src % PAGE_TOK);
          memcpy(kc4[i], hb + I4_OFF_K_CODES + slot * 128, 128);
          memcpy(sc4[i], i4_scale(hb, 0, slot), 2);
          memcpy(sc4[i] + 2, i4_scale(hb, 1, slot), 2);
          for (int c = 0; c < HEAD_DIM; ++c) vu[i][c] = (uint8_t)i4_code(hb, 1, slot, c);
        }
        for (int i = 0; i < n; ++i) {
          int64_t dst = (int64_t)ctx[s] + i;
          uint8_t* hb = head_block(&cv, s, dst, h);
          if (!hb) return ORC_BAD_PAGE;
          int slot = (int)(dst % PAGE_TOK), within = slot % TILE_TOK;
          memcpy(hb + I4_OFF_K_CODES + slot * 128, kc4[i], 128);
          memcpy(i4_scale(hb, 0, slot), sc4[i], 2);
          memcpy(i4_scale(hb, 1, slot), sc4[i] + 2, 2);
          for (int c = 0; c < HEAD_DIM; ++c) {
            uint8_t* p = hb + I4_OFF_V_CODES + (slot / TILE_TOK) * (HEAD_DIM * 32) + c * 32 + (within / 8) * 4;
            uint32_t w;
            memcpy(&w, p, 4);
            w = (w & ~(15u << i4_pos(within % 8))) | ((uint32_t)vu[i][c] << i4_pos(within % 8));
            memcpy(p, &w, 4);
          }
        }
        continue;
      }
      /* Copy every source row out first, then write: a destination slot may
       * be the source slot of a later row. */
      uint8_t kc[32][96], ks[32][16], vs[32][16], vc[32][HEAD_DIM];
      for (int i = 0; i < n; ++i) {
        int64_t src = (int64_t)ctx[s] + path[(int64_t)s * t + i];
        uint8_t* hb = head_block(&cv, s, src, h);
        if (!hb) return ORC_BAD_PAGE;
        int slot = (int)(src % PAGE_TOK);
        memcpy(kc[i], k_words(hb, slot, 0), 96);
        memcpy(ks[i], k_scale(hb, slot, 0), 16);
        for (int g = 0; g < N_GROUPS; ++g) memcpy(vs[i] + 2 * g, v_scale(hb, slot, g), 2);
        for (int c = 0; c < HEAD_DIM; ++c) {
          uint32_t w[3];
          load_words(v_words(hb, slot, c), w);
          vc[i][c] = orc_block_code(w, slot % 32);
        }
      }
      for (int i = 0; i < n; ++i) {
        int64_t dst = (int64_t)ctx[s] + i;
        uint8_t* hb = head_block(&cv, s, dst, h);
        if (!hb) return ORC_BAD_PAGE;
        int slot = (int)(dst % PAGE_TOK);
        memcpy(k_words(hb, slot, 0), kc[i], 96);
        memcpy(k_scale(hb, slot, 0), ks[i], 16);
        for (int g = 0; g < N_GROUPS; ++g) memcpy(v_scale(hb, slot, g), vs[i] + 2 * g, 2);
        for (int c = 0; c < HEAD_DIM; ++c) {
          uint32_t w[3];
          uint8_t* p = v_words(hb, slot, c);
          load_words(p, w);
          block_set_code(w, slot % 32, vc[i][c]);
          store_words(p, w);
        }
      }
    }
  }
  return ORC_OK;
}

/* Decode helpers exported for the tests. */
int orc_decode_rows(const uint8_t* pool, int64_t page_bytes, int32_t pool_pages, int32_t hkv,
                    const int32_t* page_tables, const int32_t* pt_offsets, int seq, int64_t tok_begin,
                    int64_t tok_end, int which, double* out /* [n_tok][hkv][256] */, int fmt) {
  cache_view cv = {(uint8_t*)pool, page_bytes, pool_pages, hkv, page_tables, pt_offsets};
  if (view_format(&cv, fmt) != ORC_OK) return ORC_BAD_ARG;
  for (int64_t j = tok_begin; j < tok_end; ++j)
    for (int h = 0; h < hkv; ++h) {
      int rc = decode_row(&cv, seq, j, h, which, out + ((j - tok_begin) * hkv + h) * HEAD_DIM);
      if (rc != ORC_OK) return rc;
    }
  return ORC_OK;
}

/* ------------------------------------------------------------------------
 * Lookup drafting.  Reddit posts (u/iamMess), "Now added" list, lookup-
 * augmented drafting: draft tokens are copied from earlier in the same
 * request, from where its trailing tokens (six to twelve of them) last
 * appeared before; syv-ai README (mirror), SPEC=dflash2 section: verify slots
 * past the drafter's come from the request's own context.
 *
 * Reading (the pages do not say which of 6..12 wins): lengths are tried from
 * the longest (max_len) down to the shortest (min_len); for the first length
 * L whose suffix h[n-L .. n-1] occurs earlier, at a start p < n - L (the
 * occurrence may overlap the suffix), the latest such p is taken and up to k
 * tokens h[p+L .. ] are proposed, never past the end of the history.  With no
 * occurrence at any length nothing is proposed (match_len 0, match_pos -1).
 * Written as that definition: every length, every start, every token
 * compared.
 */
int orc_lookup_draft(const int32_t* h, int64_t n, int min_len, int max_len, int k, int32_t* n_prop, int32_t* prop,
                     int32_t* match_len, int64_t* match_pos) {
  if (min_len < 1 || max_len < min_len || k < 0) return -1;
  *n_prop = 0;
  *match_len = 0;
  *match_pos = -1;
  for (int L = max_len; L >= min_len; --L) {
    if ((int64_t)L >= n) continue;  /* the suffix needs an earlier start */
    for (int64_t p = n - L - 1; p >= 0; --p) {
      int same = 1;
      for (int i = 0; i < L; ++i)
        if (h[p + i] != h[n - L + i]) { same = 0; break; }
      if (same) {
        int64_t avail = n - (p + L);
        int cnt = (int)(avail < k ? avail : k);
        for (int j = 0; j < cnt; ++j) prop[j] = h[p + L + j];
        *n_prop = cnt;
        *match_len = L;
        *match_pos = p;
        return 0;
      }
    }
  }
  return 0;
}
