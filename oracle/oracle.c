/*
 * Oracle for the quantized decode step -- TEST INFRASTRUCTURE ONLY.
 * (Only tests/, the smoke check and the bench's CPU-baseline leg use it.)
 *
 * Plain loops, one definition per function, written from the pages:
 *   [Magnitude] "Magnitude: on-device AI-agent inference engine" (0539edu.com)
 *   [Core]      "5. Core modules: format, runtime, scheduling, memory and routing"
 *               (ai-infra.cypggs.com)
 *   [TFLite]    "TFLite memory planner" (pwwt.cn)
 * Where the pages leave a step open, the reading taken is stated at the
 * function. Build with -ffp-contract=off: every fp32 step below is one
 * rounded IEEE operation, never a fused multiply-add.
 */
#include "oracle.h"

#include <math.h>
#include <omp.h>
#include <stdlib.h>
#include <string.h>

/* Threads of the parallel loops below (the row loops of the GEMVs and the
 * LM head, the per-layer store loop, the per-head attention loop); n < 1
 * restores every available core. Returns the count now in use. */
int orc_set_threads(int n) {
  omp_set_num_threads(n >= 1 ? n : omp_get_num_procs());
  return omp_get_max_threads();
}

/* ========================================================================== fp16 */

/* IEEE binary16 from a double, one rounding to nearest even. Written from
 * the binary16 format (1 sign, 5 exponent bits biased by 15, 10 fraction
 * bits; subnormals in units of 2^-24). */
uint16_t orc_f64_to_f16(double d) {
  uint64_t x;
  memcpy(&x, &d, 8);
  uint16_t sign = (uint16_t)((x >> 48) & 0x8000u);
  uint64_t frac = x & 0xFFFFFFFFFFFFFull;
  int e64 = (int)((x >> 52) & 0x7FF);
  if (e64 == 0x7FF) return (uint16_t)(sign | 0x7C00u | (frac ? 0x200u : 0u));
  if (e64 == 0) return sign; /* double subnormals are far below 2^-25 */
  uint64_t m = frac | (1ull << 52);
  int e = e64 - 1023;
  if (e >= 16) return (uint16_t)(sign | 0x7C00u);
  if (e >= -14) {
    uint64_t h = ((uint64_t)(e + 15) << 10) | ((m >> 42) & 0x3FFu);
    uint64_t rem = m & ((1ull << 42) - 1), half = 1ull << 41;
    if (rem > half || (rem == half && (h & 1))) h++;
    if (h >= 0x7C00u) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | h);
  }
  int shift = 28 - e; /* value / 2^-24 = m * 2^(e - 52 + 24) */
  if (shift > 53) return sign;
  uint64_t k = m >> shift;
  uint64_t rem = m & ((1ull << shift) - 1), half = 1ull << (shift - 1);
  if (rem > half || (rem == half && (k & 1))) k++;
  return (uint16_t)(sign | k);
}

uint16_t orc_f32_to_f16(float f) { return orc_f64_to_f16((double)f); }

float orc_f16_to_f32(uint16_t h) {
  int sign = h >> 15, e = (h >> 10) & 0x1F, f = h & 0x3FF;
  double v;
  if (e == 0x1F) return f ? NAN : (sign ? -INFINITY : INFINITY);
  if (e == 0) v = ldexp((double)f, -24);
  else v = ldexp((double)(f | 0x400), e - 25);
  return (float)(sign ? -v : v);
}

void orc_f32_to_f16_array(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(x[i]);
}

static double h2d(uint16_t h) { return (double)orc_f16_to_f32(h); }

/* ========================================================================== 4-bit weights */

/* [Core] 5.1 "quantisation": weights at 4 bits with FP16 activations (W4A16).
 * The pages name the format family but not its bytes; reading used here:
 *   - groups of 32 consecutive elements along a row; a row of n_cols values
 *     has ceil(n_cols/32) groups, the last one ragged when 32 does not divide
 *     n_cols (its statistics cover its real elements, its padding codes are 0);
 *   - per group lo = min, hi = max (fp32), min m = fp16(lo),
 *     scale s = fp16((hi - lo) / 15) with an fp32 subtract and IEEE divide;
 *   - s == 0: every code is 0; else q = clamp(rint((x - m) / s), 0, 15) in
 *     fp32 (IEEE divide, round half to even);
 *   - byte j of a group holds q[2j] in its low nibble and q[2j+1] in its high
 *     nibble, so a group is 16 bytes and a row 16 * ceil(n_cols/32) bytes;
 *   - the (scale, min) pairs are fp16 [n_rows][ceil(n_cols/32)][2]. */
static int64_t n_groups(int64_t n_cols) { return (n_cols + 31) / 32; }

static void w4_quantize_row(const float* w, int64_t n_cols, uint8_t* packed_row, uint16_t* sm_row) {
  for (int64_t g = 0; g < n_groups(n_cols); ++g) {
    const float* x = w + g * 32;
    int n = (int)(n_cols - g * 32 < 32 ? n_cols - g * 32 : 32);
    float lo = x[0], hi = x[0];
    for (int i = 1; i < n; ++i) {
      if (x[i] < lo) lo = x[i];
      if (x[i] > hi) hi = x[i];
    }
    float range = hi - lo;
    float s_exact = range / 15.0f;
    uint16_t s16 = orc_f32_to_f16(s_exact);
    uint16_t m16 = orc_f32_to_f16(lo);
    float s = orc_f16_to_f32(s16), m = orc_f16_to_f32(m16);
    int q[32] = {0};
    for (int i = 0; i < n; ++i) {
      if (s == 0.0f) {
        q[i] = 0;
      } else {
        float t = (x[i] - m) / s;
        int v = (int)rintf(t);
        q[i] = v < 0 ? 0 : (v > 15 ? 15 : v);
      }
    }
    uint8_t* out = packed_row + g * 16;
    for (int j = 0; j < 16; ++j) out[j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
    sm_row[g * 2 + 0] = s16;
    sm_row[g * 2 + 1] = m16;
  }
}

void orc_w4g32_quantize(const float* w, int64_t n_rows, int64_t n_cols, uint8_t* packed, uint16_t* sm) {
  int64_t ng = n_groups(n_cols);
#pragma omp parallel for schedule(static) if (n_rows > 1)
  for (int64_t r = 0; r < n_rows; ++r)
    w4_quantize_row(w + r * n_cols, n_cols, packed + r * ng * 16, sm + r * ng * 2);
}

/* w' = s * q + m, one fp32 multiply then one fp32 add. */
static void w4_dequant_row(const uint8_t* packed_row, const uint16_t* sm_row, int64_t n_cols, float* out) {
  for (int64_t c = 0; c < n_cols; ++c) {
    uint8_t b = packed_row[c / 2];
    int q = (c & 1) ? (b >> 4) : (b & 15);
    float s = orc_f16_to_f32(sm_row[(c / 32) * 2 + 0]);
    float m = orc_f16_to_f32(sm_row[(c / 32) * 2 + 1]);
    float sq = s * (float)q;
    out[c] = sq + m;
  }
}

void orc_w4g32_dequant(const uint8_t* packed, const uint16_t* sm, int64_t n_rows, int64_t n_cols, float* out) {
  int64_t ng = n_groups(n_cols);
#pragma omp parallel for schedule(static) if (n_rows > 1)
  for (int64_t r = 0; r < n_rows; ++r)
    w4_dequant_row(packed + r * ng * 16, sm + r * ng * 2, n_cols, out + r * n_cols);
}

/* y[t][r] = sum_c w'[r][c] * x[t][c], accumulated in double (the A16
 * contract: fp16 activations times dequantised weights). */
void orc_w4_gemv(const uint8_t* packed, const uint16_t* sm, int64_t n_rows, int64_t n_cols, int n_tok,
                 const uint16_t* x_f16, double* y) {
  int64_t ng = n_groups(n_cols);
  double* xd = (double*)malloc(sizeof(double) * n_cols * n_tok);
  for (int64_t i = 0; i < n_cols * n_tok; ++i) xd[i] = h2d(x_f16[i]);
#pragma omp parallel
  {
    float* row = (float*)malloc(sizeof(float) * n_cols);
#pragma omp for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
      w4_dequant_row(packed + r * ng * 16, sm + r * ng * 2, n_cols, row);
      for (int t = 0; t < n_tok; ++t) {
        double acc = 0.0;
        const double* xt = xd + (int64_t)t * n_cols;
        for (int64_t c = 0; c < n_cols; ++c) acc += (double)row[c] * xt[c];
        y[(int64_t)t * n_rows + r] = acc;
      }
    }
    free(row);
  }
  free(xd);
}

/* The same product by the per-group identity sum(s*q + m)x = s*sum(q x) + m*sum(x)
 * (exact in real arithmetic; in double it differs from orc_w4_gemv only by
 * rounding). A second route to the same definition, used to pin the first. */
void orc_w4_gemv_folded(const uint8_t* packed, const uint16_t* sm, int64_t n_rows, int64_t n_cols,
                        const uint16_t* x_f16, double* y) {
  int64_t ng = n_groups(n_cols);
  for (int64_t r = 0; r < n_rows; ++r) {
    double acc = 0.0;
    for (int64_t g = 0; g < ng; ++g) {
      double sqx = 0.0, sx = 0.0;
      for (int64_t c = g * 32; c < g * 32 + 32 && c < n_cols; ++c) {
        uint8_t b = packed[r * ng * 16 + c / 2];
        int q = (c & 1) ? (b >> 4) : (b & 15);
        double x = h2d(x_f16[c]);
        sqx += q * x;
        sx += x;
      }
      acc += h2d(sm[(r * ng + g) * 2 + 0]) * sqx + h2d(sm[(r * ng + g) * 2 + 1]) * sx;
    }
    y[r] = acc;
  }
}

/* ========================================================================== KV quantisers */

/* INT8 KV, one fp16 scale per (token, head) vector ([Core] 5.4 counts INT8
 * KV at one byte per value). Reading: symmetric, s = fp16(max|x| / 127),
 * q = clamp(rint(x / s), -127, 127) in fp32; s == 0 gives q = 0. */
void orc_kv_quant_int8(const uint16_t* x_f16, int n_vec, int d, int8_t* q, uint16_t* scale) {
  for (int v = 0; v < n_vec; ++v) {
    const uint16_t* x = x_f16 + (int64_t)v * d;
    float a = 0.0f;
    for (int i = 0; i < d; ++i) {
      float t = fabsf(orc_f16_to_f32(x[i]));
      if (t > a) a = t;
    }
    float s_exact = a / 127.0f;
    uint16_t s16 = orc_f32_to_f16(s_exact);
    float s = orc_f16_to_f32(s16);
    for (int i = 0; i < d; ++i) {
      int c = 0;
      if (s != 0.0f) {
        float t = orc_f16_to_f32(x[i]) / s;
        c = (int)rintf(t);
        c = c < -127 ? -127 : (c > 127 ? 127 : c);
      }
      q[(int64_t)v * d + i] = (int8_t)c;
    }
    scale[v] = s16;
  }
}

/* INT4 KV ([Core] 5.4 counts it at half a byte per value): the 4-bit
 * group-32 format of the weights applied along head_dim of each vector. */
void orc_kv_quant_int4(const uint16_t* x_f16, int n_vec, int d, uint8_t* packed, uint16_t* sm) {
  float* tmp = (float*)malloc(sizeof(float) * d);
  for (int v = 0; v < n_vec; ++v) {
    for (int i = 0; i < d; ++i) tmp[i] = orc_f16_to_f32(x_f16[(int64_t)v * d + i]);
    w4_quantize_row(tmp, d, packed + (int64_t)v * (d / 2), sm + (int64_t)v * (d / 32) * 2);
  }
  free(tmp);
}

/* ========================================================================== block pool */

/* [Core] 5.2: the KV pool is preallocated. Reading of its layout: 16-token
 * blocks; one block id covers every layer; the bytes of (layer l, block b)
 * start at (l * P + b) * BLK and hold, in order, K data [Hkv][16][d],
 * V data [Hkv][16][d], K meta [Hkv][16], V meta [Hkv][16]. Data elements are
 * 2 / 1 / 0.5 bytes (FP16 / INT8 / INT4, INT4 nibbles as in the weight
 * format), meta per (token, head) is nothing / one fp16 scale / d/32 fp16
 * (scale, min) pairs. */
static int64_t data_bytes_per_vec(int d, int dt) { return dt == ORC_KV_FP16 ? 2 * d : (dt == ORC_KV_INT8 ? d : d / 2); }
static int64_t meta_bytes_per_vec(int d, int dt) { return dt == ORC_KV_FP16 ? 0 : (dt == ORC_KV_INT8 ? 2 : (d / 32) * 4); }

int64_t orc_kv_block_bytes(int hkv, int d, int dt, int bt) {
  return 2 * (int64_t)hkv * bt * (data_bytes_per_vec(d, dt) + meta_bytes_per_vec(d, dt));
}

/* part: 0 K data, 1 V data, 2 K meta, 3 V meta. */
int64_t orc_kv_offset(int hkv, int d, int dt, int bt, int64_t pool_blocks, int layer, int64_t block, int part,
                      int head, int slot) {
  int64_t base = ((int64_t)layer * pool_blocks + block) * orc_kv_block_bytes(hkv, d, dt, bt);
  int64_t db = data_bytes_per_vec(d, dt), mb = meta_bytes_per_vec(d, dt);
  int64_t data_part = (int64_t)hkv * bt * db, meta_part = (int64_t)hkv * bt * mb;
  int64_t vec = (int64_t)head * bt + slot;
  switch (part) {
    case 0: return base + vec * db;
    case 1: return base + data_part + vec * db;
    case 2: return base + 2 * data_part + vec * mb;
    default: return base + 2 * data_part + meta_part + vec * mb;
  }
}

/* [Core] 5.4 "KV capacity planning": KV per token = 2 x layers x KV heads x
 * head_dim x bytes per value. */
int64_t orc_kv_bytes_per_token(int n_layers, int n_kv_heads, int head_dim, double bytes_per_value) {
  return (int64_t)(2.0 * n_layers * n_kv_heads * head_dim * bytes_per_value);
}

/* [Core] 5.4: max context = (total memory - OS reserve - weights) / KV per token. */
int64_t orc_kv_max_context(double total, double os, double weights, double bpt) {
  return (int64_t)floor((total - os - weights) / bpt);
}

/* ========================================================================== arena planner */

/* [TFLite] 2.1: a tensor lives from its producer to its last consumer; with
 * closed intervals [first, last] two tensors may share bytes only if one's
 * last op comes strictly before the other's first (an op reads its inputs
 * while it writes its output). closed_intervals = 0 gives the half-open
 * reading [first, last) used only to check the page's worked example.
 * [TFLite] 2.2: place tensors largest first (ties: earlier first op, then
 * lower id), each at the lowest offset, rounded up to `align` ([TFLite] 2.2:
 * 64-byte starts), where it overlaps no already-placed tensor whose lifetime
 * overlaps its own. Returns the arena size, rounded up to `align`. */
static int live_overlap(int f1, int l1, int f2, int l2, int closed) {
  return closed ? (f1 <= l2 && f2 <= l1) : (f1 < l2 && f2 < l1);
}

static int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

int64_t orc_arena_plan(int n, const int64_t* size, const int* first, const int* last, int64_t align,
                       int closed, int64_t* offset) {
  int* order = (int*)malloc(sizeof(int) * (n > 0 ? n : 1));
  for (int i = 0; i < n; ++i) order[i] = i;
  /* insertion sort: size desc, first asc, id asc */
  for (int i = 1; i < n; ++i) {
    int t = order[i], j = i - 1;
    while (j >= 0) {
      int o = order[j];
      int before = size[t] > size[o] || (size[t] == size[o] && (first[t] < first[o] || (first[t] == first[o] && t < o)));
      if (!before) break;
      order[j + 1] = o;
      --j;
    }
    order[j + 1] = t;
  }
  int* placed = (int*)malloc(sizeof(int) * (n > 0 ? n : 1));
  int n_placed = 0;
  int* cand = (int*)malloc(sizeof(int) * (n > 0 ? n : 1));
  int64_t arena = 0;
  for (int oi = 0; oi < n; ++oi) {
    int t = order[oi];
    int nc = 0;
    for (int k = 0; k < n_placed; ++k) {
      int p = placed[k];
      if (live_overlap(first[t], last[t], first[p], last[p], closed)) cand[nc++] = p;
    }
    /* sort the overlapping placed tensors by (offset, end) */
    for (int i = 1; i < nc; ++i) {
      int x = cand[i], j = i - 1;
      while (j >= 0) {
        int y = cand[j];
        int before = offset[x] < offset[y] || (offset[x] == offset[y] && offset[x] + size[x] < offset[y] + size[y]);
        if (!before) break;
        cand[j + 1] = y;
        --j;
      }
      cand[j + 1] = x;
    }
    int64_t cur = 0;
    for (int i = 0; i < nc; ++i) {
      int p = cand[i];
      if (align_up(cur, align) + size[t] <= offset[p]) break;
      if (offset[p] + size[p] > cur) cur = offset[p] + size[p];
    }
    offset[t] = align_up(cur, align);
    if (offset[t] + size[t] > arena) arena = offset[t] + size[t];
    placed[n_placed++] = t;
  }
  free(order);
  free(placed);
  free(cand);
  return align_up(arena, align);
}

/* ========================================================================== layer pieces */

/* RMSNorm ahead of attention and FFN ([Core] 5.1 "pre-norm"); reading:
 * xn_i = fp16(r_i / sqrt(mean(r^2) + eps) * gamma_i). */
void orc_rmsnorm(const double* r, const uint16_t* gamma, int n, float eps, uint16_t* out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += r[i] * r[i];
  double inv = 1.0 / sqrt(ss / n + (double)eps);
  for (int i = 0; i < n; ++i) out[i] = orc_f64_to_f16(r[i] * inv * h2d(gamma[i]));
}

/* [Core] 5.1 "rope table pre-generation". Reading: rotate-half pairing
 * (i, i + d/2), angle p * base^(-2i/d) computed in double, cos and sin in
 * double, stored as fp32. Row p holds d/2 entries. */
void orc_rope_table(int max_pos, int head_dim, float base, float* cos_out, float* sin_out) {
  int half = head_dim / 2;
  for (int p = 0; p < max_pos; ++p)
    for (int i = 0; i < half; ++i) {
      double theta = (double)p * pow((double)base, -2.0 * i / head_dim);
      cos_out[(int64_t)p * half + i] = (float)cos(theta);
      sin_out[(int64_t)p * half + i] = (float)sin(theta);
    }
}

/* x'_i = x_i c - x_{i+d/2} s ; x'_{i+d/2} = x_i s + x_{i+d/2} c, rounded to fp16. */
void orc_rope_apply(const uint16_t* x, int head_dim, const float* cos_row, const float* sin_row, uint16_t* out) {
  int half = head_dim / 2;
  uint16_t* tmp = (uint16_t*)malloc(sizeof(uint16_t) * head_dim);
  for (int i = 0; i < half; ++i) {
    double a = h2d(x[i]), b = h2d(x[i + half]), c = cos_row[i], s = sin_row[i];
    tmp[i] = orc_f64_to_f16(a * c - b * s);
    tmp[i + half] = orc_f64_to_f16(a * s + b * c);
  }
  memcpy(out, tmp, sizeof(uint16_t) * head_dim);
  free(tmp);
}

/* ========================================================================== logical KV store */

struct orc_kv {
  orc_cfg cfg;
  int cap, len;
  /* per layer, per which (0 K, 1 V): token-major [cap][Hkv] vectors */
  uint8_t** data; /* [L*2] -> [cap][Hkv][data bytes] */
  uint8_t** meta; /* [L*2] -> [cap][Hkv][meta bytes] */
};

orc_kv* orc_kv_create(const orc_cfg* cfg, int capacity) {
  orc_kv* kv = (orc_kv*)calloc(1, sizeof(orc_kv));
  kv->cfg = *cfg;
  kv->cap = capacity;
  int L = cfg->n_layers, H = cfg->n_kv_heads, d = cfg->head_dim, dt = cfg->kv_dtype;
  kv->data = (uint8_t**)calloc(2 * L, sizeof(uint8_t*));
  kv->meta = (uint8_t**)calloc(2 * L, sizeof(uint8_t*));
  for (int i = 0; i < 2 * L; ++i) {
    kv->data[i] = (uint8_t*)calloc((size_t)capacity * H * data_bytes_per_vec(d, dt), 1);
    int64_t mb = meta_bytes_per_vec(d, dt);
    kv->meta[i] = mb ? (uint8_t*)calloc((size_t)capacity * H * mb, 1) : NULL;
  }
  return kv;
}

void orc_kv_destroy(orc_kv* kv) {
  if (!kv) return;
  for (int i = 0; i < 2 * kv->cfg.n_layers; ++i) {
    free(kv->data[i]);
    free(kv->meta[i]);
  }
  free(kv->data);
  free(kv->meta);
  free(kv);
}

int orc_kv_len(const orc_kv* kv) { return kv->len; }

/* Forget every token from position len on (bookkeeping only). */
void orc_kv_truncate(orc_kv* kv, int len) {
  if (len >= 0 && len <= kv->len) kv->len = len;
}

/* Tokens that orc_layer stored past the length (a pass run layer by layer)
 * become part of the store: len += n. Returns 0, or -1 past the capacity. */
int orc_kv_commit(orc_kv* kv, int n) {
  if (n < 0 || kv->len + n > kv->cap) return -1;
  kv->len += n;
  return 0;
}

/* Store one fp16 vector of head_dim values in the configured KV precision. */
static void kv_store_vec(orc_kv* kv, int layer, int which, int tok, int head, const uint16_t* x) {
  int H = kv->cfg.n_kv_heads, d = kv->cfg.head_dim, dt = kv->cfg.kv_dtype;
  int64_t db = data_bytes_per_vec(d, dt), mb = meta_bytes_per_vec(d, dt);
  int64_t vec = (int64_t)tok * H + head;
  uint8_t* dst = kv->data[layer * 2 + which] + vec * db;
  if (dt == ORC_KV_FP16) {
    memcpy(dst, x, (size_t)db);
  } else if (dt == ORC_KV_INT8) {
    uint16_t s;
    orc_kv_quant_int8(x, 1, d, (int8_t*)dst, &s);
    memcpy(kv->meta[layer * 2 + which] + vec * mb, &s, 2);
  } else {
    uint16_t sm[64];
    orc_kv_quant_int4(x, 1, d, dst, sm);
    memcpy(kv->meta[layer * 2 + which] + vec * mb, sm, (size_t)mb);
  }
}

int orc_kv_append(orc_kv* kv, int n_tok, const uint16_t* k, const uint16_t* v) {
  int L = kv->cfg.n_layers, H = kv->cfg.n_kv_heads, d = kv->cfg.head_dim;
  if (kv->len + n_tok > kv->cap) return -1;
#pragma omp parallel for schedule(static)
  for (int l = 0; l < L; ++l)
    for (int t = 0; t < n_tok; ++t)
      for (int h = 0; h < H; ++h) {
        int64_t src = (((int64_t)l * n_tok + t) * H + h) * d;
        kv_store_vec(kv, l, 0, kv->len + t, h, k + src);
        kv_store_vec(kv, l, 1, kv->len + t, h, v + src);
      }
  kv->len += n_tok;
  return 0;
}

/* Dequantised stored vector: FP16 as stored, INT8 q*s, INT4 s*q + m (fp32). */
void orc_kv_read(const orc_kv* kv, int layer, int which, int tok, int head, float* out) {
  int H = kv->cfg.n_kv_heads, d = kv->cfg.head_dim, dt = kv->cfg.kv_dtype;
  int64_t db = data_bytes_per_vec(d, dt), mb = meta_bytes_per_vec(d, dt);
  int64_t vec = (int64_t)tok * H + head;
  const uint8_t* src = kv->data[layer * 2 + which] + vec * db;
  if (dt == ORC_KV_FP16) {
    const uint16_t* h = (const uint16_t*)src;
    for (int i = 0; i < d; ++i) out[i] = orc_f16_to_f32(h[i]);
  } else if (dt == ORC_KV_INT8) {
    uint16_t s16;
    memcpy(&s16, kv->meta[layer * 2 + which] + vec * mb, 2);
    float s = orc_f16_to_f32(s16);
    for (int i = 0; i < d; ++i) out[i] = (float)((const int8_t*)src)[i] * s;
  } else {
    const uint16_t* sm = (const uint16_t*)(kv->meta[layer * 2 + which] + vec * mb);
    w4_dequant_row(src, sm, d, out);
  }
}

int64_t orc_kv_stored(const orc_kv* kv, int layer, int which, int tok, int head, uint8_t* data, uint8_t* meta) {
  int H = kv->cfg.n_kv_heads, d = kv->cfg.head_dim, dt = kv->cfg.kv_dtype;
  int64_t db = data_bytes_per_vec(d, dt), mb = meta_bytes_per_vec(d, dt);
  int64_t vec = (int64_t)tok * H + head;
  memcpy(data, kv->data[layer * 2 + which] + vec * db, (size_t)db);
  if (mb && meta) memcpy(meta, kv->meta[layer * 2 + which] + vec * mb, (size_t)mb);
  return db;
}

/* Softmax attention of one query head over keys 0..n_keys-1 of its KV head:
 * score_t = q . k_t / sqrt(d), softmax with the max subtracted, o = sum w_t v_t,
 * all in double over the dequantised stored K and V; o rounded to fp16. */
void orc_attention(const orc_cfg* cfg, const orc_kv* kv, int layer, int kv_head, const uint16_t* q_f16, int n_keys,
                   uint16_t* out_f16) {
  int d = cfg->head_dim;
  double* score = (double*)malloc(sizeof(double) * (n_keys > 0 ? n_keys : 1));
  float* vec = (float*)malloc(sizeof(float) * d);
  double* acc = (double*)calloc(d, sizeof(double));
  double mx = -INFINITY;
  for (int t = 0; t < n_keys; ++t) {
    orc_kv_read(kv, layer, 0, t, kv_head, vec);
    double s = 0.0;
    for (int i = 0; i < d; ++i) s += h2d(q_f16[i]) * (double)vec[i];
    score[t] = s / sqrt((double)d);
    if (score[t] > mx) mx = score[t];
  }
  double l = 0.0;
  for (int t = 0; t < n_keys; ++t) {
    double w = exp(score[t] - mx);
    l += w;
    orc_kv_read(kv, layer, 1, t, kv_head, vec);
    for (int i = 0; i < d; ++i) acc[i] += w * (double)vec[i];
  }
  for (int i = 0; i < d; ++i) out_f16[i] = orc_f64_to_f16(acc[i] / l);
  free(score);
  free(vec);
  free(acc);
}

/* ========================================================================== whole step */

/* Positions of the T tokens of a pass: sequence s appends n_tok[s] tokens at
 * len_s .. len_s + n_tok[s] - 1 (tokens ordered sequence by sequence).
 * Returns T, or -1 if a store or the RoPE table is too short. */
static int token_positions(int n_seq, orc_kv* const* kv, const int* n_tok, int rope_rows, int** seq_of, int** pos) {
  int T = 0;
  for (int s = 0; s < n_seq; ++s) {
    if (kv[s]->len + n_tok[s] > kv[s]->cap || kv[s]->len + n_tok[s] > rope_rows) return -1;
    T += n_tok[s];
  }
  *seq_of = (int*)malloc(sizeof(int) * (T > 0 ? T : 1));
  *pos = (int*)malloc(sizeof(int) * (T > 0 ? T : 1));
  for (int s = 0, t = 0; s < n_seq; ++s)
    for (int i = 0; i < n_tok[s]; ++i, ++t) {
      (*seq_of)[t] = s;
      (*pos)[t] = kv[s]->len + i;
    }
  return T;
}

/* One layer of the pre-norm GQA decoder ([Core] 5.1: pre-norm, merged QKV,
 * merged gate-up, precomputed RoPE table; [Core] 5.2: KV pool written in
 * place) for n_seq sequences, sequence s appending n_tok[s] tokens at
 * positions len_s .. len_s + n_tok[s] - 1 with causal attention. For every
 * token, from its residual r (double):
 *   xn = rmsnorm(r, gamma1)                          fp16
 *   [q; k; v] = W_qkv xn                             fp16
 *   q, k rotated at the token's position             fp16
 *   k, v stored in the KV store at this layer (quantised there)
 *   o_h = attention(q_h, keys 0..p of KV head h/G)   fp16   (h/G: contiguous grouping)
 *   r += W_o o
 *   xn2 = rmsnorm(r, gamma2)                         fp16
 *   [g; u] = W_gu xn2,  a = silu(g) * u              fp16
 *   r += W_down a
 * r_in and r_out are [T][D] (they may be the same array); the stores'
 * lengths are not advanced (the pass's last layer is followed by that).
 * Returns 0, or -1 if a store is full or the RoPE table is too short. */
int orc_layer(const orc_cfg* cfg, const orc_weights* w, int l, int n_seq, orc_kv* const* kv, const int* n_tok,
              const double* r_in, const float* rope_cos, const float* rope_sin, int rope_rows, double* r_out) {
  int D = cfg->hidden, Hq = cfg->n_heads, Hkv = cfg->n_kv_heads, d = cfg->head_dim;
  int F = cfg->ffn, G = Hq / Hkv, half = d / 2;
  int R = (Hq + 2 * Hkv) * d;
  int *seq_of = NULL, *pos = NULL;
  int T = token_positions(n_seq, kv, n_tok, rope_rows, &seq_of, &pos);
  if (T < 0) return -1;
  double* r = r_out;
  if (r != r_in) memcpy(r, r_in, sizeof(double) * (size_t)T * D);
  uint16_t* xn = (uint16_t*)malloc(sizeof(uint16_t) * T * D);
  double* y = (double*)malloc(sizeof(double) * (int64_t)T * (R > 2 * F ? R : 2 * F));
  uint16_t* qkv = (uint16_t*)malloc(sizeof(uint16_t) * (int64_t)T * R);
  uint16_t* o = (uint16_t*)malloc(sizeof(uint16_t) * (int64_t)T * Hq * d);
  uint16_t* a = (uint16_t*)malloc(sizeof(uint16_t) * (int64_t)T * F);

  for (int t = 0; t < T; ++t) orc_rmsnorm(r + (int64_t)t * D, w->gamma1[l], D, cfg->rms_eps, xn + (int64_t)t * D);
  orc_w4_gemv(w->wqkv[l], w->sqkv[l], R, D, T, xn, y);
  for (int64_t i = 0; i < (int64_t)T * R; ++i) qkv[i] = orc_f64_to_f16(y[i]);
  for (int t = 0; t < T; ++t) {
    const float* c = rope_cos + (int64_t)pos[t] * half;
    const float* sn = rope_sin + (int64_t)pos[t] * half;
    uint16_t* row = qkv + (int64_t)t * R;
    for (int h = 0; h < Hq + Hkv; ++h) orc_rope_apply(row + h * d, d, c, sn, row + h * d);
    for (int h = 0; h < Hkv; ++h) {
      kv_store_vec(kv[seq_of[t]], l, 0, pos[t], h, row + (Hq + h) * d);
      kv_store_vec(kv[seq_of[t]], l, 1, pos[t], h, row + (Hq + Hkv + h) * d);
    }
  }
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < Hq; ++h)
      orc_attention(cfg, kv[seq_of[t]], l, h / G, qkv + (int64_t)t * R + h * d, pos[t] + 1,
                    o + ((int64_t)t * Hq + h) * d);
  orc_w4_gemv(w->wo[l], w->so[l], D, Hq * d, T, o, y);
  for (int64_t i = 0; i < (int64_t)T * D; ++i) r[i] += y[i];
  for (int t = 0; t < T; ++t) orc_rmsnorm(r + (int64_t)t * D, w->gamma2[l], D, cfg->rms_eps, xn + (int64_t)t * D);
  orc_w4_gemv(w->wgu[l], w->sgu[l], 2 * F, D, T, xn, y);
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < F; ++j) {
      double g = y[(int64_t)t * 2 * F + j], u = y[(int64_t)t * 2 * F + F + j];
      a[(int64_t)t * F + j] = orc_f64_to_f16(g / (1.0 + exp(-g)) * u);
    }
  orc_w4_gemv(w->wdown[l], w->sdown[l], D, F, T, a, y);
  for (int64_t i = 0; i < (int64_t)T * D; ++i) r[i] += y[i];
  free(seq_of);
  free(pos);
  free(xn);
  free(y);
  free(qkv);
  free(o);
  free(a);
  return 0;
}

/* Output of one token from its final residual r [D] (double): the fp16 logits
 * W_lm xf with xf = rmsnorm(r, gamma_f) (fp16), accumulated in double and
 * rounded once, [V]; or fp16(r) [D] when the model has no LM head. */
void orc_output(const orc_cfg* cfg, const orc_weights* w, const double* r, uint16_t* out_f16) {
  int D = cfg->hidden, V = cfg->vocab;
  if (V == 0) {
    for (int i = 0; i < D; ++i) out_f16[i] = orc_f64_to_f16(r[i]);
    return;
  }
  uint16_t* xf = (uint16_t*)malloc(sizeof(uint16_t) * D);
  orc_rmsnorm(r, w->gamma_f, D, cfg->rms_eps, xf);
  double* xd = (double*)malloc(sizeof(double) * D);
  for (int i = 0; i < D; ++i) xd[i] = h2d(xf[i]);
#pragma omp parallel for schedule(static)
  for (int v = 0; v < V; ++v) {
    const uint16_t* row = w->lm_head + (int64_t)v * D;
    double acc = 0.0;
    for (int i = 0; i < D; ++i) acc += h2d(row[i]) * xd[i];
    out_f16[v] = orc_f64_to_f16(acc);
  }
  free(xd);
  free(xf);
}

/* The whole pass: the residual r of every token starts as its fp16 input and
 * is carried unrounded through orc_layer for layers 0..L-1; then every store
 * has grown by its n_tok, and the output of the last token of each sequence
 * s goes to out_f16[s] (orc_output: [V], or [D] without an LM head). n_tok = 1
 * for every sequence is the decode step; one sequence with n_tok = T is a
 * prefill chunk. Returns 0, or -1 if a store is full or the RoPE table is too
 * short (nothing is stored then). */
int orc_forward(const orc_cfg* cfg, const orc_weights* w, int n_seq, orc_kv* const* kv, const int* n_tok,
                const uint16_t* x_f16, const float* rope_cos, const float* rope_sin, int rope_rows,
                uint16_t* out_f16) {
  int D = cfg->hidden, V = cfg->vocab;
  int *seq_of = NULL, *pos = NULL;
  int T = token_positions(n_seq, kv, n_tok, rope_rows, &seq_of, &pos);
  if (T < 0) return -1;
  free(seq_of);
  free(pos);
  double* r = (double*)malloc(sizeof(double) * (size_t)T * D);
  for (int64_t i = 0; i < (int64_t)T * D; ++i) r[i] = h2d(x_f16[i]);
  for (int l = 0; l < cfg->n_layers; ++l) orc_layer(cfg, w, l, n_seq, kv, n_tok, r, rope_cos, rope_sin, rope_rows, r);
  for (int s = 0; s < n_seq; ++s) kv[s]->len += n_tok[s];
  int64_t width = V ? V : D;
  for (int s = 0, t_last = -1; s < n_seq; ++s) {
    t_last += n_tok[s];
    orc_output(cfg, w, r + (int64_t)t_last * D, out_f16 + (int64_t)s * width);
  }
  free(r);
  return 0;
}
