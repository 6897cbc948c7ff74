/*
 * okc_oracle.c — plain, slow CPU oracle of the paged-FP8 gated attention block.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library. It shares no code, header,
 * table or constant generator with the CUDA library.
 *
 * What it computes follows "012-attention-local-splits.py" (the SGLang Muse
 * Spark attention problem file): the `_prepare_qkv` kernel, `_cos_sin`, the
 * flash_attn_with_kvcache arguments and the rms_norm_gate call. It applies each
 * step literally, token by token and head by head; attention runs in double
 * precision over every visible key, with no splits, tiles or reordering.
 *
 * Readings taken where the page is silent (each also listed in the design notes):
 *  - float -> bf16 and float -> E4M3 are round-to-nearest-even; E4M3 saturates to
 *    +-448 (satfinite) and keeps the sign of zero; NaN encodes as 0x7F|sign.
 *  - The RMS inverse is the float32 rounding of the exact 1/sqrt(sum(x^2)/64 + eps),
 *    eps being the float32 constant 1e-5 of the kernel.
 *  - Each float32 product and sum of the RoPE rotation is rounded separately
 *    (no fused multiply-add); this file is compiled with -ffp-contract=off.
 *  - theta^e, 1/x, cos and sin of the RoPE table are float32 roundings of the
 *    exact values (libm in double, rounded once).
 *  - The attention output is rounded to bf16 once (FA3 returns bf16) before the
 *    norm-gate; the norm-gate is evaluated in double and rounded once to bf16.
 *  - q_norm 1 (the vLLM CuTeDSL `qk_norm` page, `QKNormDirectKernel.kernel` and
 *    the `qk_norm(x, head_dim, eps, scale)` wrapper): a q head is x * rstd times
 *    the output scale, both products float32 operations, and the store to bf16
 *    is its only rounding to bf16; the output scale is the query factor
 *    (qk_scale_factor), so it leaves the softmax scale, which is then sm_scale
 *    alone. k heads are normed with scale 1, which is the q_norm 0 arithmetic.
 *
 * Every function works on plain arrays; bf16 values travel as uint16 bit patterns,
 * E4M3 values as uint8 codes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_D 64

/* ---------------------------------------------------------------- formats */

/* Round v to a binary floating-point format with p significant bits and minimum
 * normal exponent emin, to nearest, ties to even (no overflow handling). This is
 * the plain definition: the quantum is 2^(max(e, emin) - (p-1)) where e is the
 * exponent of v's leading bit. */
static double round_to_format(double v, int p, int emin) {
  if (v == 0.0 || !isfinite(v)) return v;
  int e;
  frexp(fabs(v), &e); /* |v| = f * 2^e, f in [0.5, 1): leading bit at e-1 */
  int lead = e - 1;
  if (lead < emin) lead = emin;
  double q = ldexp(1.0, lead - (p - 1));
  return rint(v / q) * q; /* v/q is exact; rint rounds half to even */
}

/* bf16: 8 significant bits, emin -126. */
double orc_bf16_round(double v) {
  if (isnan(v)) return v;
  double r = round_to_format(v, 8, -126);
  if (fabs(r) > 3.3895313892515355e38) r = copysign(INFINITY, v); /* beyond max bf16 */
  return r;
}

uint16_t orc_bf16_bits(double v) {
  float f = (float)orc_bf16_round(v); /* exact: a bf16 value is a float value */
  uint32_t u;
  memcpy(&u, &f, 4);
  if (isnan(v)) return (uint16_t)(0x7FC0u | ((u >> 16) & 0x8000u));
  return (uint16_t)(u >> 16);
}

double orc_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* E4M3 (OCP FP8 e4m3fn): bias 7, 3 mantissa bits, subnormal quantum 2^-9, largest
 * finite 448, no infinities, NaN = S.1111.111. */
double orc_e4m3_value(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double a;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    a = ldexp((double)m, -9);
  else
    a = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -a : a;
}

uint8_t orc_e4m3_code(double v) {
  if (isnan(v)) return (uint8_t)(0x7Fu | (signbit(v) ? 0x80u : 0u));
  uint8_t sign = signbit(v) ? 0x80u : 0u;
  double r = fabs(round_to_format(v, 4, -6));
  if (r > 448.0) r = 448.0; /* satfinite */
  if (r == 0.0) return sign;
  int e;
  frexp(r, &e);
  int lead = e - 1;
  uint8_t code;
  if (lead < -6) {
    code = (uint8_t)ldexp(r, 9); /* subnormal: r = m * 2^-9 */
  } else {
    int mant = (int)((ldexp(r, -lead) - 1.0) * 8.0);
    code = (uint8_t)(((lead + 7) << 3) | mant);
  }
  return (uint8_t)(code | sign);
}

void orc_bf16_round_array(const double* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = orc_bf16_bits(in[i]);
}

void orc_e4m3_code_array(const double* in, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = orc_e4m3_code(in[i]);
}

void orc_e4m3_value_array(const uint8_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = orc_e4m3_value(in[i]);
}

/* ------------------------------------------------------------------- RoPE */

/* `_cos_sin`: inv_freq = 1 / theta^(arange(0, d, 2)/d) in float32. */
void orc_rope_inv_freq(float theta, float* inv_freq /* [32] */) {
  for (int i = 0; i < ORC_D / 2; i++) {
    float e = (float)(2 * i) / (float)ORC_D;                 /* exact */
    float pw = (float)pow((double)theta, (double)e);       /* float32 power */
    inv_freq[i] = 1.0f / pw;                               /* float32 division */
  }
}

/* Row `pos` of the [2^21, 64] table: cos(pos*inv_freq) | sin(pos*inv_freq). */
void orc_rope_row(float theta, int64_t pos, float* cos_out /* [32] */, float* sin_out /* [32] */) {
  float inv[ORC_D / 2];
  orc_rope_inv_freq(theta, inv);
  for (int i = 0; i < ORC_D / 2; i++) {
    float ang = (float)pos * inv[i]; /* float32 outer product, one rounding */
    cos_out[i] = (float)cos((double)ang);
    sin_out[i] = (float)sin((double)ang);
  }
}

/* ---------------------------------------------------- steps 1-3: prepare */

typedef struct orc_cfg {
  int32_t batch, q_len, hq, hkv, page_size, window, max_pages, num_pages;
  float rope_theta, qk_scale_factor, sm_scale, kv_scale;
  int32_t q_norm; /* 0: the problem file's norm; 1: the vLLM qk_norm with the query factor folded in */
} orc_cfg;

/*
 * `_prepare_qkv` for all T tokens. k_cache / v_cache are updated in place at
 * cache_loc rows; q8 receives [T, Hq, 64] E4M3 codes. Rows outside the pool are
 * skipped and counted in the return value (never written).
 */
int64_t orc_prepare(const orc_cfg* cfg, int64_t T, const uint16_t* qkv, const int64_t* positions,
                    const int64_t* cache_loc, uint8_t* k_cache, uint8_t* v_cache, float k_scale,
                    float v_scale, uint8_t* q8) {
  const int hq = cfg->hq, hkv = cfg->hkv, heads = hq + 2 * hkv;
  const int width = (2 * hq + 2 * hkv) * ORC_D;
  const int rope = cfg->rope_theta != 0.0f;
  const int scaled = cfg->kv_scale != 1.0f;
  const int64_t rows = (int64_t)cfg->num_pages * cfg->page_size;
  const float eps = 1.0e-5f;
  int64_t skipped = 0;
  float cs[ORC_D / 2], sn[ORC_D / 2];

  for (int64_t t = 0; t < T; t++) {
    const uint16_t* row = qkv + t * width;
    const int64_t slot = cache_loc[t];
    const int slot_ok = slot >= 0 && slot < rows;
    if (!slot_ok) skipped++;
    if (rope) orc_rope_row(cfg->rope_theta, positions[t], cs, sn);
    for (int h = 0; h < heads; h++) {
      float x[ORC_D], y[ORC_D], out[ORC_D];
      for (int c = 0; c < ORC_D; c++) x[c] = (float)orc_bf16_value(row[h * ORC_D + c]);
      if (h < hq + hkv) {
        /* RMSNorm: float32 inverse of the exact root mean square, then bf16. */
        double sumsq = 0.0;
        for (int c = 0; c < ORC_D; c++) sumsq += (double)x[c] * (double)x[c];
        float inv = (float)(1.0 / sqrt(sumsq / ORC_D + (double)eps));
        if (h < hq && cfg->q_norm == 1) {
          /* float32 x * rstd, float32 times the output scale, one bf16 rounding */
          for (int c = 0; c < ORC_D; c++) {
            const float normed = x[c] * inv;
            const float scaled_q = normed * cfg->qk_scale_factor;
            y[c] = (float)orc_bf16_round((double)scaled_q);
          }
        } else {
          for (int c = 0; c < ORC_D; c++) y[c] = (float)orc_bf16_round((double)(x[c] * inv));
        }
        if (rope) {
          /* Interleaved pairs (2i, 2i+1) share angle i; the partner of column c
           * is column c^1, normalised and rounded like y. */
          for (int c = 0; c < ORC_D; c++) {
            float p = y[c ^ 1], co = cs[c / 2], si = sn[c / 2];
            float a = y[c] * co, b = p * si;
            float r = (c % 2 == 0) ? a - b : a + b;
            out[c] = (float)orc_bf16_round((double)r);
          }
        } else {
          memcpy(out, y, sizeof out);
        }
        if (h < hq) {
          for (int c = 0; c < ORC_D; c++)
            q8[(t * hq + h) * ORC_D + c] = orc_e4m3_code((double)out[c]);
        } else if (slot_ok) {
          for (int c = 0; c < ORC_D; c++) {
            float key = out[c];
            if (scaled) key = (float)orc_bf16_round((double)(key / k_scale));
            k_cache[(slot * hkv + (h - hq)) * ORC_D + c] = orc_e4m3_code((double)key);
          }
        }
      } else if (slot_ok) {
        for (int c = 0; c < ORC_D; c++) {
          float value = x[c];
          if (scaled) value = (float)orc_bf16_round((double)(value / v_scale));
          v_cache[(slot * hkv + (h - hq - hkv)) * ORC_D + c] = orc_e4m3_code((double)value);
        }
      }
    }
  }
  return skipped;
}

/* -------------------------------------------------------- step 4: attention */

/*
 * flash_attn_with_kvcache(causal=True, window_size=(window-1, 0) or (-1,-1)),
 * written as the definition: for query row (t, h) at position p, the keys are
 * j in [lo, p] with lo = max(0, p - window + 1) (window > 0) or 0; key j of
 * request b is the cache row page_table[b][j / P] * P + j % P; the logit is
 * (q . K_j) * softmax_scale with K_j = E4M3 value * k_scale (scaled path) and
 * o = sum_j softmax_j V_j, V_j = E4M3 value * v_scale (scaled path).
 * The softmax scale is the float32 value of sm_scale * qk_scale_factor, or of
 * sm_scale alone under q_norm 1 (the factor is then inside q).
 *
 * Only rows with mask[t*Hq + h] != 0 are computed (mask NULL = all rows).
 * o: double [T, Hq, 64]; lse (may be NULL): natural log-sum-exp of the logits.
 * Returns the number of visible keys whose page id was invalid (read as zeros).
 */
int64_t orc_attention(const orc_cfg* cfg, const uint8_t* q8, const uint8_t* k_cache,
                      const uint8_t* v_cache, float k_scale, float v_scale,
                      const int32_t* page_table, const int32_t* cache_seqlens,
                      const int32_t* cu_seqlens_q, const uint8_t* mask, double* o, double* lse) {
  const int hq = cfg->hq, hkv = cfg->hkv, group = hq / hkv, P = cfg->page_size;
  const int scaled = cfg->kv_scale != 1.0f;
  const double ks = scaled ? (double)k_scale : 1.0, vs = scaled ? (double)v_scale : 1.0;
  const double scale = cfg->q_norm == 1 ? (double)cfg->sm_scale
                                         : (double)(float)((double)cfg->sm_scale * (double)cfg->qk_scale_factor);
  int64_t bad = 0;
  double val[256]; /* decoded E4M3 codes, so the loops below are plain multiply-adds */
  for (int c = 0; c < 256; c++) val[c] = orc_e4m3_value((uint8_t)c);

  for (int b = 0; b < cfg->batch; b++) {
    const int64_t n = cache_seqlens[b];
    const int64_t ql = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
    for (int64_t i = 0; i < ql; i++) {
      const int64_t t = cu_seqlens_q[b] + i;
      const int64_t p = n - ql + i;
      const int64_t lo = cfg->window > 0 ? (p - cfg->window + 1 > 0 ? p - cfg->window + 1 : 0) : 0;
      const int64_t nk = p - lo + 1;
      for (int h = 0; h < hq; h++) {
        if (mask && !mask[t * hq + h]) continue;
        const int g = h / group;
        double qv[ORC_D];
        for (int c = 0; c < ORC_D; c++) qv[c] = val[q8[(t * hq + h) * ORC_D + c]];
        double* s = (double*)malloc((size_t)(nk > 0 ? nk : 1) * sizeof(double));
        int64_t* rowid = (int64_t*)malloc((size_t)(nk > 0 ? nk : 1) * sizeof(int64_t));
        double mx = -INFINITY;
        for (int64_t j = lo; j <= p; j++) {
          const int64_t page = page_table[(int64_t)b * cfg->max_pages + j / P];
          int64_t r = -1;
          if (j / P < cfg->max_pages && page >= 0 && page < cfg->num_pages)
            r = page * P + j % P;
          else
            bad++;
          rowid[j - lo] = r;
          double dot = 0.0;
          if (r >= 0)
            for (int c = 0; c < ORC_D; c++)
              dot += qv[c] * (val[k_cache[(r * hkv + g) * ORC_D + c]] * ks);
          s[j - lo] = dot * scale;
          if (s[j - lo] > mx) mx = s[j - lo];
        }
        double denom = 0.0, acc[ORC_D];
        for (int c = 0; c < ORC_D; c++) acc[c] = 0.0;
        for (int64_t j = 0; j < nk; j++) {
          const double w = exp(s[j] - mx);
          denom += w;
          if (rowid[j] >= 0)
            for (int c = 0; c < ORC_D; c++)
              acc[c] += w * (val[v_cache[(rowid[j] * hkv + g) * ORC_D + c]] * vs);
        }
        for (int c = 0; c < ORC_D; c++) o[(t * hq + h) * ORC_D + c] = acc[c] / denom;
        if (lse) lse[t * hq + h] = mx + log(denom);
        free(s);
        free(rowid);
      }
    }
  }
  return bad;
}

/* ------------------------------------------------------ step 5: norm-gate */

/*
 * rms_norm_gate(out.to(bf16), gate, weight, eps, has_norm=True), per head of 64:
 * ob = bf16(o); out = bf16(ob / sqrt(mean(ob^2) + eps) * w * sigmoid(gate)),
 * evaluated in double and rounded once. weight: bf16 [64] or NULL (None = 1).
 * gate rows are read from qkv at column (Hq + 2Hkv)*64 + h*64 + c.
 */
void orc_normgate(const orc_cfg* cfg, int64_t T, const double* o, const uint16_t* qkv,
                  const uint16_t* weight, float eps, const uint8_t* mask, uint16_t* out) {
  const int hq = cfg->hq, hkv = cfg->hkv;
  const int width = (2 * hq + 2 * hkv) * ORC_D, gate0 = (hq + 2 * hkv) * ORC_D;
  for (int64_t t = 0; t < T; t++) {
    for (int h = 0; h < hq; h++) {
      if (mask && !mask[t * hq + h]) continue;
      double ob[ORC_D], ms = 0.0;
      for (int c = 0; c < ORC_D; c++) {
        ob[c] = orc_bf16_round(o[(t * hq + h) * ORC_D + c]);
        ms += ob[c] * ob[c];
      }
      ms /= ORC_D;
      const double r = 1.0 / sqrt(ms + (double)eps);
      for (int c = 0; c < ORC_D; c++) {
        const double g = orc_bf16_value(qkv[t * width + gate0 + h * ORC_D + c]);
        const double w = weight ? orc_bf16_value(weight[c]) : 1.0;
        const double sig = 1.0 / (1.0 + exp(-g));
        out[(t * hq + h) * ORC_D + c] = orc_bf16_bits(ob[c] * r * w * sig);
      }
    }
  }
}
