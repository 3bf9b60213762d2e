/*
 * The step before decode attention for one layer, as a plain fp64 CPU oracle:
 * per-head RMS normalisation of the new token's q, k and v, rotary position
 * embedding of q and k at the token's position, and the paged-cache slot its
 * k / v rows go to.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call, link or
 * load this file; only the tests use it. It shares no code, header or table
 * with the CUDA path.
 *
 * Sources (page title, section):
 *   - Gemma 4 layers normalise q, k and v per head and then apply RoPE, and
 *     both are fused with the write of the new token into the paged KV cache:
 *     Sparse-vLLM PR #27 "feat: support Gemma 4 and native multimodal
 *     inference", section "专用算子与性能优化" (dedicated operators: QKV norm +
 *     RoPE); the vLLM concepts page "模型库与算子层 — 概念", section on compile
 *     fusion passes (norm / RoPE folded into the paged KV-cache write);
 *   - sliding-window and global layers carry their own RoPE parameters and
 *     their own RoPE cache: PR #27, section "Gemma 4 文本推理" (text inference);
 *   - the paged KV cache and its [num_pages, Hkv, P, d] slice: the vLLM concepts
 *     page, section "注意力层" (attention layer).
 *
 * Readings where the pages are silent:
 *   - the new token's position is pos = L_b - 1, L_b counting the cached tokens
 *     including the new one (the decode oracle's length);
 *   - RMS normalisation of a head vector x with weight w:
 *       y_i = x_i / sqrt(mean_j x_j^2 + eps) * w_i
 *     (a model whose norm scales by 1 + w passes 1 + w as the weight); v has
 *     its own weight, unit when none is given;
 *   - RoPE rotates the first `rot` dims (rot even, rot <= d) in pairs
 *     (i, i + rot/2), i < rot/2, by the angle pos * theta^(-2i/rot):
 *       y_i        <- y_i cos a - y_{i+rot/2} sin a
 *       y_{i+rot/2} <- y_{i+rot/2} cos a + y_i sin a
 *     and leaves dims >= rot unchanged; theta and rot are the layer's own;
 *   - on a layer that stores K=V the cached row is the normalised, rotated k
 *     (v is not used);
 *   - the new rows go to page block_table[b][pos / P], row pos % P.
 *
 * All arithmetic is IEEE fp64 from the exact bf16 inputs. Build with
 * -ffp-contract=off so x86 and Arm hosts produce identical bits.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define REF_OK 0
#define REF_BAD_ARG -1
#define REF_BAD_LEN -3

static double prep_bf16_to_f64(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* y = x / sqrt(mean(x^2) + eps) * w ; w == NULL means unit weight. */
static void rms_norm(const uint16_t *x, const uint16_t *w, int d, double eps, double *y) {
  double ms = 0.0;
  for (int i = 0; i < d; ++i) {
    const double v = prep_bf16_to_f64(x[i]);
    ms += v * v;
  }
  const double r = 1.0 / sqrt(ms / d + eps);
  for (int i = 0; i < d; ++i) y[i] = prep_bf16_to_f64(x[i]) * r * (w ? prep_bf16_to_f64(w[i]) : 1.0);
}

/* Angle of pair i at position pos: pos * theta^(-2i/rot). */
static double rope_angle(int pos, int i, int rot, double theta) {
  return (double)pos * pow(theta, -2.0 * i / rot);
}

/* Rotate the pairs (i, i + rot/2) of y in place. */
static void rope(double *y, int rot, int pos, double theta) {
  const int half = rot / 2;
  for (int i = 0; i < half; ++i) {
    const double a = rope_angle(pos, i, rot, theta);
    const double c = cos(a), s = sin(a);
    const double x1 = y[i], x2 = y[i + half];
    y[i] = x1 * c - x2 * s;
    y[i + half] = x2 * c + x1 * s;
  }
}

/*
 * The RoPE table of one layer: out[p * rot + i] = cos(angle(p, i)) and
 * out[p * rot + rot/2 + i] = sin(angle(p, i)), p < n_pos, i < rot/2.
 */
int ref_rope_table(int rot, double theta, int n_pos, double *out) {
  if (rot < 2 || rot % 2 || n_pos < 0 || !(theta > 0.0) || !out) return REF_BAD_ARG;
  const int half = rot / 2;
  for (int p = 0; p < n_pos; ++p)
    for (int i = 0; i < half; ++i) {
      const double a = rope_angle(p, i, rot, theta);
      out[(size_t)p * rot + i] = cos(a);
      out[(size_t)p * rot + half + i] = sin(a);
    }
  return REF_OK;
}

/*
 * For every request b (pos = L_b - 1):
 *   q_out[b, h] = rope(rms_norm(q_in[b, h], q_w), pos)   h < Hq
 *   k_out[b, g] = rope(rms_norm(k_in[b, g], k_w), pos)   g < Hkv
 *   v_out[b, g] = rms_norm(v_in[b, g], v_w)               (not on a K=V layer)
 *   slot_page[b] = block_tables[b][pos / P] (-1 when outside the pool),
 *   slot_row[b]  = pos % P.
 * q_in [B, Hq, d], k_in / v_in [B, Hkv, d] and the weights [d] are bf16 bit
 * patterns; outputs are fp64 of the same shapes. rot = 0 skips the rotation.
 * Returns REF_BAD_LEN if some L_b is outside [1, max_pages * P].
 */
int ref_prepare_qkv(int B, int Hq, int Hkv, int d, int P, int num_pages, int max_pages, int kv_shared, int rot,
                    double theta, double eps, const uint16_t *q_in, const uint16_t *k_in, const uint16_t *v_in,
                    const uint16_t *q_w, const uint16_t *k_w, const uint16_t *v_w, const int32_t *block_tables,
                    const int32_t *seq_lens, double *q_out, double *k_out, double *v_out, int32_t *slot_page,
                    int32_t *slot_row) {
  if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || d < 1 || P < 1 || num_pages < 0 || max_pages < 0) return REF_BAD_ARG;
  if (rot < 0 || rot % 2 || rot > d || (rot > 0 && !(theta > 0.0)) || eps < 0.0) return REF_BAD_ARG;
  if (!q_in || !k_in || !q_w || !k_w || !seq_lens || !q_out || !k_out || !slot_page || !slot_row) return REF_BAD_ARG;
  if (!kv_shared && (!v_in || !v_out)) return REF_BAD_ARG;
  for (int b = 0; b < B; ++b) {
    const int L = seq_lens[b];
    if (L < 1 || (long long)L > (long long)max_pages * P) return REF_BAD_LEN;
  }
  for (int b = 0; b < B; ++b) {
    const int pos = seq_lens[b] - 1;
    for (int h = 0; h < Hq; ++h) {
      double *y = q_out + ((size_t)b * Hq + h) * d;
      rms_norm(q_in + ((size_t)b * Hq + h) * d, q_w, d, eps, y);
      rope(y, rot, pos, theta);
    }
    for (int g = 0; g < Hkv; ++g) {
      double *y = k_out + ((size_t)b * Hkv + g) * d;
      rms_norm(k_in + ((size_t)b * Hkv + g) * d, k_w, d, eps, y);
      rope(y, rot, pos, theta);
      if (!kv_shared) rms_norm(v_in + ((size_t)b * Hkv + g) * d, v_w, d, eps, v_out + ((size_t)b * Hkv + g) * d);
    }
    const int page = block_tables[(size_t)b * max_pages + pos / P];
    slot_page[b] = (page >= 0 && page < num_pages) ? page : -1;
    slot_row[b] = pos % P;
  }
  return REF_OK;
}
