/*
 * CPU oracle for the attention step of a Qwen2 decoder layer over a
 * block-paged KV cache.  TEST INFRASTRUCTURE ONLY: it is linked by the tests,
 * by the smoke check and by the CPU-baseline leg of the benchmark, never by
 * the CUDA path, and it shares no code with it.
 *
 * Plain, slow, obviously correct: fp64 arithmetic over the bf16 values the
 * GPU sees, explicit loops, no blocking or fusion.  Build with
 * -ffp-contract=off so the fp32 RoPE recipe below is evaluated as written.
 *
 * Sources (the pages this restates):
 *   [p1] "Qwen2 模型结构代码详解" (lpnh.cn/news/2488257), section 2 "配置解析":
 *        rope_theta defaults to 1000000, head_dim = hidden // heads = 128,
 *        scaling = head_dim ** -0.5, 28 Q heads share 4 KV heads (7 per group).
 *   [p2] "Qwen2大模型架构解析与vLLM优化实践", section 2.2 (get_rope(head_dim,
 *        rotary_dim=head_dim, max_position, base=rope_theta)) and section 4.1
 *        (Attention(num_heads, head_dim, scaling, num_kv_heads, cache_config)).
 *   [p3] vLLM-deploys-Qwen notes (gsyq.cn/news/2022324), section 2.1:
 *        PagedAttention keeps the KV cache in fixed-size blocks.
 *   [p4] Qwen engineering notes (0539edu.com/news/4254669), section 2.1:
 *        FlashAttention-2 varlen (packed variable-length) causal attention.
 *   [p5] nano-vllm Qwen3 skeleton (adg.csdn.net), section 5: per-sequence
 *        block_table, prepare_prefill/set_context supply slots and positions.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes of the repository):
 *   - cache layout [num_blocks][Hkv][BS][D]; slot = block * BS + offset;
 *   - query head h uses KV head h / (H / Hkv) (consecutive grouping);
 *   - rotate-half pairs dimension i with i + D/2 over the full head_dim;
 *   - the cos/sin table is cos/sin(pos * theta^(-2i/D)) in fp64, rounded to
 *     fp32; the rotation is done in fp32 with every product and sum rounded
 *     (no fused multiply-add), then rounded to bf16 nearest-even;
 *   - a negative slot is a padding token: nothing is written;
 *   - chunked prefill is bottom-right aligned: query i of a sequence with
 *     q_len new tokens and context L sits at position L - q_len + i and sees
 *     keys 0 .. L - q_len + i;
 *   - a row whose context is invalid, or whose block id is out of range,
 *     is written as zeros and an error bit is returned;
 *   - an FP8 cache ([p2] sections 4.1-4.2 and 6.3: kv_cache_dtype "fp8",
 *     fp8_e4m3fn, a cache scale per tensor) holds the e4m3fn code of
 *     x / scale for the bf16 value x a bf16 cache would hold (fp32 division,
 *     then round-to-nearest-even, saturating to +-448); attention reads
 *     code * scale.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Error bits, shared meaning with the library's device error word. */
#define OR_ERR_SLOT 1
#define OR_ERR_BLOCK 2
#define OR_ERR_CONTEXT 4
#define OR_ERR_POSITION 16
/* oracle only: an RMSNorm sum of squares was not exact in fp64 */
#define OR_ERR_NORM_INEXACT 64

/* ---------------------------------------------------------------- bf16 --- */

static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static double bf16_to_f64(uint16_t b) { return (double)bf16_to_f32(b); }

/* Round-to-nearest-even of an fp32 value to bf16 (NaN kept quiet). */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

uint16_t oracle_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }
double oracle_bf16_to_f64(uint16_t b) { return bf16_to_f64(b); }

/* ---------------------------------------------------------- e4m3fn ---- */

/* The OCP 8-bit float E4M3 ("fn": finite, no infinities): sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits.  Exponent field 0 holds the
 * subnormals m * 2^-9; field e > 0 holds (1 + m/8) * 2^(e-7); the codes
 * S.1111.111 are NaN, so the largest finite value is 1.75 * 2^8 = 448. */
double oracle_e4m3_to_f64(uint8_t c) {
  const int e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return (c & 0x80) ? -mag : mag;
}

/* Rounds v / 2^q to an integer, ties to even (v >= 0, exact in double). */
static double round_half_even_scaled(double v, int q) {
  const double x = ldexp(v, -q);
  const double f = floor(x);
  const double r = x - f;
  if (r > 0.5) return f + 1.0;
  if (r < 0.5) return f;
  return fmod(f, 2.0) == 0.0 ? f : f + 1.0;
}

/* fp32 -> e4m3fn code, round to nearest even, saturating: a magnitude that
 * rounds above 448 (and an infinity) gives the largest finite code; NaN
 * gives 0x7F. */
uint8_t oracle_f32_to_e4m3(float f) {
  if (f != f) return 0x7F;
  const uint8_t sign = signbit(f) ? 0x80 : 0x00;
  const double a = fabs((double)f);
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    /* subnormal grid: multiples of 2^-9 (8 of them reach 2^-6, the first
     * normal, code 0x08) */
    const double m = round_half_even_scaled(a, -9);
    return sign | (uint8_t)m;
  }
  int ex;
  frexp(a, &ex);          /* a = fr * 2^ex, fr in [0.5, 1) */
  int E = ex - 1;         /* a in [2^E, 2^(E+1)) */
  double mm = round_half_even_scaled(a - ldexp(1.0, E), E - 3);  /* eighths */
  if (mm == 8.0) {
    mm = 0.0;
    ++E;
  }
  if (E > 8 || (E == 8 && mm > 6.0)) return sign | 0x7E;
  return sign | (uint8_t)(((E + 7) << 3) | (int)mm);
}

void oracle_f32_to_e4m3_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_e4m3(x[i]);
}

void oracle_e4m3_to_f64_array(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_to_f64(c[i]);
}

/* The cache code of a bf16 value x under a per-tensor scale: e4m3(x / s),
 * the division in fp32 (correctly rounded). */
static uint8_t quantize_kv(uint16_t x, float s) {
  const float q = bf16_to_f32(x) / s;
  return oracle_f32_to_e4m3(q);
}

/* ------------------------------------------------------- RoPE table ---- */

/* [p2] section 2.2 get_rope(head_dim, rotary_dim=head_dim, max_position,
 * base): one row per position 0 .. max_pos-1; columns 0 .. D/2-1 hold
 * cos(pos * theta^(-2i/D)), columns D/2 .. D-1 the matching sin. */
int oracle_rope_table(double theta, int32_t max_pos, int32_t head_dim,
                      float* cos_sin) {
  if (max_pos <= 0 || head_dim <= 0 || (head_dim & 1) || !(theta > 0.0))
    return -1;
  const int32_t half = head_dim / 2;
  for (int32_t pos = 0; pos < max_pos; ++pos) {
    for (int32_t i = 0; i < half; ++i) {
      double inv_freq = pow(theta, -(2.0 * (double)i) / (double)head_dim);
      double angle = (double)pos * inv_freq;
      cos_sin[(int64_t)pos * head_dim + i] = (float)cos(angle);
      cos_sin[(int64_t)pos * head_dim + half + i] = (float)sin(angle);
    }
  }
  return 0;
}

/* RoPE tables with rope_scaling ("Qwen2大模型架构解析与vLLM优化实践" section
 * 7.1, rope_scaling {type, factor, original_max_position}):
 *   scaling 0: none (the table above);
 *   scaling 1: linear -- positions divided by factor, angle = (pos/factor) *
 *              theta^(-2i/D);
 *   scaling 2: dynamic NTK -- the base is raised when the table must cover
 *              more than original_max positions: for max_pos > original_max,
 *              base = theta * (factor * max_pos / original_max - (factor - 1))
 *              ^ (D / (D - 2)), else base = theta; angle = pos * base^(-2i/D).
 *              The table's max_pos plays the current sequence-length bound
 *              ("dynamic": a longer batch rebuilds its table).
 * Angles in fp64, cos and sin rounded to fp32. */
int oracle_rope_table_scaled(double theta, int32_t max_pos, int32_t head_dim,
                             int32_t scaling, double factor, int32_t original_max,
                             float* cos_sin) {
  if (max_pos <= 0 || head_dim <= 2 || (head_dim & 1) || !(theta > 0.0)) return -1;
  if (scaling < 0 || scaling > 2) return -1;
  if (scaling != 0 && !(factor >= 1.0)) return -1;
  if (scaling == 2 && original_max <= 0) return -1;
  const int32_t half = head_dim / 2;
  double base = theta;
  if (scaling == 2 && max_pos > original_max) {
    double s = factor * (double)max_pos / (double)original_max - (factor - 1.0);
    base = theta * pow(s, (double)head_dim / (double)(head_dim - 2));
  }
  for (int32_t pos = 0; pos < max_pos; ++pos) {
    double p = scaling == 1 ? (double)pos / factor : (double)pos;
    for (int32_t i = 0; i < half; ++i) {
      double inv_freq = pow(base, -(2.0 * (double)i) / (double)head_dim);
      double angle = p * inv_freq;
      cos_sin[(int64_t)pos * head_dim + i] = (float)cos(angle);
      cos_sin[(int64_t)pos * head_dim + half + i] = (float)sin(angle);
    }
  }
  return 0;
}

/* ------------------------------------------------------- RoPE apply ---- */

/* Rotate-half on one head vector, fp32 recipe: for i < D/2,
 *   y[i]       = x[i]       * c_i - x[i+D/2] * s_i
 *   y[i+D/2]   = x[i+D/2]   * c_i + x[i]     * s_i
 * each product and each sum rounded to fp32, result rounded to bf16. */
void oracle_rope_head_exact(const uint16_t* x, int32_t head_dim,
                            const float* cos_sin_row, uint16_t* y) {
  const int32_t half = head_dim / 2;
  for (int32_t i = 0; i < half; ++i) {
    float x1 = bf16_to_f32(x[i]);
    float x2 = bf16_to_f32(x[i + half]);
    float c = cos_sin_row[i];
    float s = cos_sin_row[half + i];
    float a = x1 * c;
    float b = x2 * s;
    float lo = a - b;
    float d = x2 * c;
    float e = x1 * s;
    float hi = d + e;
    y[i] = f32_to_bf16_rne(lo);
    y[i + half] = f32_to_bf16_rne(hi);
  }
}

/* The same rotation in fp64 with exact angles (no table), on fp64 input. */
void oracle_rope_head_f64(const double* x, int32_t head_dim, double pos,
                          double theta, double* y) {
  const int32_t half = head_dim / 2;
  for (int32_t i = 0; i < half; ++i) {
    double inv_freq = pow(theta, -(2.0 * (double)i) / (double)head_dim);
    double c = cos(pos * inv_freq), s = sin(pos * inv_freq);
    y[i] = x[i] * c - x[i + half] * s;
    y[i + half] = x[i + half] * c + x[i] * s;
  }
}

/* ---------------------------------------------------- cache append ---- */

/* Rotate q in place and write rotated k and raw v into the paged caches.
 * q/k/v rows are strided (elements); head h of row t starts at
 * row + h * head_dim.  Returns OR-ed error bits. */
int32_t oracle_rope_cache_append(
    uint16_t* q, int64_t q_row_stride, const uint16_t* k, int64_t k_row_stride,
    const uint16_t* v, int64_t v_row_stride, const int32_t* positions,
    const int32_t* slot_mapping, int32_t num_tokens, uint16_t* k_cache,
    uint16_t* v_cache, int32_t num_blocks, const float* cos_sin,
    int32_t max_pos, int32_t num_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size) {
  int32_t err = 0;
  uint16_t* tmp = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)head_dim);
  for (int32_t t = 0; t < num_tokens; ++t) {
    int32_t pos = positions[t];
    if (pos < 0 || pos >= max_pos) {
      err |= OR_ERR_POSITION;
      continue;
    }
    const float* row = cos_sin + (int64_t)pos * head_dim;
    for (int32_t h = 0; h < num_heads; ++h) {
      uint16_t* qh = q + (int64_t)t * q_row_stride + (int64_t)h * head_dim;
      oracle_rope_head_exact(qh, head_dim, row, tmp);
      memcpy(qh, tmp, sizeof(uint16_t) * (size_t)head_dim);
    }
    int32_t slot = slot_mapping[t];
    if (slot < 0) continue; /* padding token */
    if ((int64_t)slot >= (int64_t)num_blocks * block_size) {
      err |= OR_ERR_SLOT;
      continue;
    }
    int32_t blk = slot / block_size, off = slot % block_size;
    for (int32_t g = 0; g < num_kv_heads; ++g) {
      int64_t dst = (((int64_t)blk * num_kv_heads + g) * block_size + off) *
                    head_dim;
      const uint16_t* kh = k + (int64_t)t * k_row_stride + (int64_t)g * head_dim;
      const uint16_t* vh = v + (int64_t)t * v_row_stride + (int64_t)g * head_dim;
      oracle_rope_head_exact(kh, head_dim, row, k_cache + dst);
      memcpy(v_cache + dst, vh, sizeof(uint16_t) * (size_t)head_dim);
    }
  }
  free(tmp);
  return err;
}

/* --------------------------- qkv bias and per-head RMSNorm (Qwen3) ---- */

/* The qkv projection's bias: "Qwen2大模型架构解析与vLLM优化实践" (qkv_proj
 * with bias=True) and the nano-vllm Qwen3 skeleton (qkv_bias from
 * attention_bias).  Reading: the biased projection output is a bf16 tensor,
 * x' = bf16(float(x) + float(b)) -- one rounding (the fp32 sum of two bf16
 * values is exact unless their exponents differ by more than 16). */
void oracle_add_bias_head(const uint16_t* x, const uint16_t* b, int32_t n, uint16_t* y) {
  for (int32_t i = 0; i < n; ++i) {
    float s = bf16_to_f32(x[i]) + bf16_to_f32(b[i]);
    y[i] = f32_to_bf16_rne(s);
  }
}

/* RMSNorm of one head vector with a per-dimension weight (the Qwen3
 * attention's q_norm / k_norm, nano-vllm Qwen3 skeleton page, module tree;
 * eps = rms_norm_eps): y_i = x_i / sqrt(mean(x^2) + eps) * w_i.  The page
 * names the module, not its rounding.  Reading: a bf16 tensor operation
 * around an exact mean square --
 *   ss = the exact sum of the squares of the n bf16 values.  It is summed
 *        in fp64 in index order: a bf16 square has 16 significant bits, so
 *        every square and every partial sum is exact unless the head's
 *        nonzero magnitudes span more than about 2^18; the function
 *        returns 1 if any addition was rounded (the reading then does not
 *        hold), else 0;
 *   v  = fp32(ss / n + eps), one rounding, with eps taken as the fp32
 *        number the C interface passes;
 *   r  = 1 / sqrt(v), correctly rounded fp32 square root and division;
 *   y_i = bf16(fp32(fp32(x_i * r) * w_i)). */
int32_t oracle_rmsnorm_head(const uint16_t* x, const uint16_t* w, int32_t n, double eps,
                            uint16_t* y) {
  double ss = 0.0;
  int32_t inexact = 0;
  for (int32_t i = 0; i < n; ++i) {
    const double xi = bf16_to_f64(x[i]);
    const double sq = xi * xi; /* exact: 8 significant bits squared */
    const double t = ss + sq;
    if (isfinite(t)) {
      /* error of the rounded addition (Knuth's two-sum) */
      const double bv = t - ss;
      const double e = (ss - (t - bv)) + (sq - bv);
      if (e != 0.0) inexact = 1;
    }
    ss = t;
  }
  const double e32 = (double)(float)eps;
  const float v = (float)(ss / (double)n + e32);
  const float r = 1.0f / sqrtf(v);
  for (int32_t i = 0; i < n; ++i) {
    const float t = bf16_to_f32(x[i]) * r;
    const float u = t * bf16_to_f32(w[i]);
    y[i] = f32_to_bf16_rne(u);
  }
  return inexact;
}

/* oracle_rope_cache_append with the projection bias and the Qwen3 head
 * norms first: for each token, q heads: q = rope(norm_q(bias(q))); k heads:
 * k = rope(norm_k(bias(k))) into the cache; v heads: v = bias(v) into the
 * cache.  Any of bias / q_norm_w / k_norm_w may be NULL (step skipped).
 * bias: [(H + 2 Hkv) * D] (q heads, then k, then v); norm weights: [D]. */
int32_t oracle_rope_cache_append_ex(
    uint16_t* q, int64_t q_row_stride, const uint16_t* k, int64_t k_row_stride,
    const uint16_t* v, int64_t v_row_stride, const int32_t* positions,
    const int32_t* slot_mapping, int32_t num_tokens, uint16_t* k_cache,
    uint16_t* v_cache, int32_t num_blocks, const float* cos_sin,
    int32_t max_pos, int32_t num_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, const uint16_t* bias,
    const uint16_t* q_norm_w, const uint16_t* k_norm_w, double eps) {
  int32_t err = 0;
  const int32_t D = head_dim;
  uint16_t* a = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)D);
  uint16_t* b = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)D);
  for (int32_t t = 0; t < num_tokens; ++t) {
    int32_t pos = positions[t];
    if (pos < 0 || pos >= max_pos) {
      err |= OR_ERR_POSITION;
      continue;
    }
    const float* row = cos_sin + (int64_t)pos * D;
    for (int32_t h = 0; h < num_heads; ++h) {
      uint16_t* qh = q + (int64_t)t * q_row_stride + (int64_t)h * D;
      memcpy(a, qh, sizeof(uint16_t) * (size_t)D);
      if (bias) oracle_add_bias_head(a, bias + (int64_t)h * D, D, a);
      if (q_norm_w) {
        if (oracle_rmsnorm_head(a, q_norm_w, D, eps, b)) err |= OR_ERR_NORM_INEXACT;
        memcpy(a, b, sizeof(uint16_t) * (size_t)D);
      }
      oracle_rope_head_exact(a, D, row, qh);
    }
    int32_t slot = slot_mapping[t];
    if (slot < 0) continue; /* padding token */
    if ((int64_t)slot >= (int64_t)num_blocks * block_size) {
      err |= OR_ERR_SLOT;
      continue;
    }
    int32_t blk = slot / block_size, off = slot % block_size;
    for (int32_t g = 0; g < num_kv_heads; ++g) {
      int64_t dst = (((int64_t)blk * num_kv_heads + g) * block_size + off) * D;
      const uint16_t* kh = k + (int64_t)t * k_row_stride + (int64_t)g * D;
      const uint16_t* vh = v + (int64_t)t * v_row_stride + (int64_t)g * D;
      memcpy(a, kh, sizeof(uint16_t) * (size_t)D);
      if (bias) oracle_add_bias_head(a, bias + (int64_t)(num_heads + g) * D, D, a);
      if (k_norm_w) {
        if (oracle_rmsnorm_head(a, k_norm_w, D, eps, b)) err |= OR_ERR_NORM_INEXACT;
        memcpy(a, b, sizeof(uint16_t) * (size_t)D);
      }
      oracle_rope_head_exact(a, D, row, k_cache + dst);
      if (bias)
        oracle_add_bias_head(vh, bias + (int64_t)(num_heads + num_kv_heads + g) * D, D,
                             v_cache + dst);
      else
        memcpy(v_cache + dst, vh, sizeof(uint16_t) * (size_t)D);
    }
  }
  free(a);
  free(b);
  return err;
}

/* The append into an FP8 cache: every step of oracle_rope_cache_append_ex
 * up to the bf16 K (rotated) and V rows a bf16 cache would receive, then
 * each value is stored as quantize_kv(x, k_scale) / quantize_kv(x, v_scale).
 * q is rotated in place as before. */
int32_t oracle_rope_cache_append_fp8(
    uint16_t* q, int64_t q_row_stride, const uint16_t* k, int64_t k_row_stride,
    const uint16_t* v, int64_t v_row_stride, const int32_t* positions,
    const int32_t* slot_mapping, int32_t num_tokens, uint8_t* k_cache,
    uint8_t* v_cache, int32_t num_blocks, const float* cos_sin,
    int32_t max_pos, int32_t num_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, const uint16_t* bias,
    const uint16_t* q_norm_w, const uint16_t* k_norm_w, double eps,
    float k_scale, float v_scale) {
  const int32_t D = head_dim;
  /* one token at a time through the bf16 append into a one-block scratch
   * cache, then quantised */
  uint16_t* kb = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)num_kv_heads * D);
  uint16_t* vb = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)num_kv_heads * D);
  int32_t err = 0;
  for (int32_t t = 0; t < num_tokens; ++t) {
    int32_t slot = slot_mapping[t];
    const int32_t zero = 0;
    const int32_t e = oracle_rope_cache_append_ex(
        q + (int64_t)t * q_row_stride, q_row_stride, k + (int64_t)t * k_row_stride,
        k_row_stride, v + (int64_t)t * v_row_stride, v_row_stride, positions + t,
        slot < 0 ? &slot : &zero, 1, kb, vb, 1, cos_sin, max_pos, num_heads,
        num_kv_heads, D, 1, bias, q_norm_w, k_norm_w, eps);
    err |= e;
    if ((e & ~OR_ERR_NORM_INEXACT) || slot < 0) continue;
    if ((int64_t)slot >= (int64_t)num_blocks * block_size) {
      err |= OR_ERR_SLOT;
      continue;
    }
    const int32_t blk = slot / block_size, off = slot % block_size;
    for (int32_t g = 0; g < num_kv_heads; ++g) {
      const int64_t dst = (((int64_t)blk * num_kv_heads + g) * block_size + off) * D;
      for (int32_t d = 0; d < D; ++d) {
        k_cache[dst + d] = quantize_kv(kb[(int64_t)g * D + d], k_scale);
        v_cache[dst + d] = quantize_kv(vb[(int64_t)g * D + d], v_scale);
      }
    }
  }
  free(kb);
  free(vb);
  return err;
}

/* ------------------------------------------------------- attention ---- */

typedef struct attn_job_s {
  double* out;
  const uint16_t* q;
  int64_t q_row_stride;
  const int32_t* cu_seqlens_q; /* NULL: decode, one query per sequence */
  int32_t num_seqs;
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  const uint8_t* k_cache8; /* FP8 cache (k_cache / v_cache unused) or NULL */
  const uint8_t* v_cache8;
  double k_scale, v_scale;
  int32_t num_blocks;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  const int32_t* context_lens;
  int32_t num_heads, num_kv_heads, head_dim, block_size;
  double scale;
  int32_t partition_tokens; /* 0: one softmax over all keys */
  int32_t nthreads;
  int32_t next_unit; /* guarded by lock */
  int32_t err;
  pthread_mutex_t lock;
} attn_job;

/* Element i of the K or V cache as the attention sees it: the bf16 value,
 * or code * scale for an FP8 cache. */
static double k_at(const struct attn_job_s* J, int64_t i);
static double v_at(const struct attn_job_s* J, int64_t i);

/* One query row, one head.  Keys 0 .. last (inclusive) of sequence b.
 * Without partitions: o = sum_j softmax(z)_j v_j with
 * z_j = scale * q . k_j.  With partitions of P keys (the split-KV form):
 * each partition s keeps m_s = max z, l_s = sum e^(z - m_s) and
 * o_s = sum e^(z - m_s) v_j; the merge takes M = max m_s and returns
 * sum e^(m_s - M) o_s / sum e^(m_s - M) l_s. */
static int32_t attend_row(const attn_job* J, int32_t b, const uint16_t* qh,
                          int32_t g, int32_t last, double* o) {
  const int32_t D = J->head_dim, BS = J->block_size;
  const int32_t nkeys = last + 1;
  for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
  /* Gather check first: every block the row needs must be in range. */
  for (int32_t j = 0; j < nkeys; j += BS) {
    int32_t blk = J->block_tables[(int64_t)b * J->max_blocks_per_seq + j / BS];
    if (blk < 0 || blk >= J->num_blocks) return OR_ERR_BLOCK;
  }
  double* z = (double*)malloc(sizeof(double) * (size_t)nkeys);
  for (int32_t j = 0; j < nkeys; ++j) {
    int32_t blk = J->block_tables[(int64_t)b * J->max_blocks_per_seq + j / BS];
    int32_t off = j % BS;
    const int64_t kj = (((int64_t)blk * J->num_kv_heads + g) * BS + off) * D;
    double dot = 0.0;
    for (int32_t d = 0; d < D; ++d) dot += bf16_to_f64(qh[d]) * k_at(J, kj + d);
    z[j] = J->scale * dot;
  }
  const int32_t P = J->partition_tokens > 0 ? J->partition_tokens : nkeys;
  const int32_t nparts = (nkeys + P - 1) / P;
  double* m = (double*)malloc(sizeof(double) * (size_t)nparts);
  double* l = (double*)malloc(sizeof(double) * (size_t)nparts);
  double* os = (double*)calloc((size_t)nparts * D, sizeof(double));
  for (int32_t s = 0; s < nparts; ++s) {
    int32_t j0 = s * P, j1 = j0 + P < nkeys ? j0 + P : nkeys;
    double mx = -INFINITY;
    for (int32_t j = j0; j < j1; ++j) mx = z[j] > mx ? z[j] : mx;
    double sum = 0.0;
    for (int32_t j = j0; j < j1; ++j) {
      double p = exp(z[j] - mx);
      sum += p;
      int32_t blk = J->block_tables[(int64_t)b * J->max_blocks_per_seq + j / BS];
      const int64_t vj = (((int64_t)blk * J->num_kv_heads + g) * BS + j % BS) * D;
      for (int32_t d = 0; d < D; ++d) os[(int64_t)s * D + d] += p * v_at(J, vj + d);
    }
    m[s] = mx;
    l[s] = sum;
  }
  double M = -INFINITY;
  for (int32_t s = 0; s < nparts; ++s) M = m[s] > M ? m[s] : M;
  double denom = 0.0;
  for (int32_t s = 0; s < nparts; ++s) denom += exp(m[s] - M) * l[s];
  for (int32_t d = 0; d < D; ++d) {
    double num = 0.0;
    for (int32_t s = 0; s < nparts; ++s) num += exp(m[s] - M) * os[(int64_t)s * D + d];
    o[d] = num / denom;
  }
  free(z);
  free(m);
  free(l);
  free(os);
  return 0;
}

static double k_at(const attn_job* J, int64_t i) {
  return J->k_cache8 ? oracle_e4m3_to_f64(J->k_cache8[i]) * J->k_scale : bf16_to_f64(J->k_cache[i]);
}

static double v_at(const attn_job* J, int64_t i) {
  return J->v_cache8 ? oracle_e4m3_to_f64(J->v_cache8[i]) * J->v_scale : bf16_to_f64(J->v_cache[i]);
}

/* Work unit = (sequence, query head); units are handed out in order. */
static void* attn_worker(void* arg) {
  attn_job* J = (attn_job*)arg;
  const int32_t H = J->num_heads, D = J->head_dim;
  const int32_t group = H / J->num_kv_heads;
  int32_t local_err = 0;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int32_t u = J->next_unit++;
    pthread_mutex_unlock(&J->lock);
    if (u >= J->num_seqs * H) break;
    int32_t b = u / H, h = u % H, g = h / group;
    int32_t t0 = J->cu_seqlens_q ? J->cu_seqlens_q[b] : b;
    int32_t t1 = J->cu_seqlens_q ? J->cu_seqlens_q[b + 1] : b + 1;
    int32_t q_len = t1 - t0;
    int32_t L = J->context_lens[b];
    for (int32_t t = t0; t < t1; ++t) {
      double* o = J->out + ((int64_t)t * H + h) * D;
      const uint16_t* qh = J->q + (int64_t)t * J->q_row_stride + (int64_t)h * D;
      int32_t last = L - q_len + (t - t0); /* bottom-right causal alignment */
      if (L <= 0 || q_len <= 0 || q_len > L ||
          L > J->max_blocks_per_seq * J->block_size) {
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        local_err |= OR_ERR_CONTEXT;
        continue;
      }
      int32_t e = attend_row(J, b, qh, g, last, o);
      if (e) {
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        local_err |= e;
      }
    }
  }
  pthread_mutex_lock(&J->lock);
  J->err |= local_err;
  pthread_mutex_unlock(&J->lock);
  return NULL;
}

/* Paged GQA attention for decode (cu_seqlens_q == NULL: query row b belongs
 * to sequence b) and for causal varlen / chunked prefill (query rows
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 belong to sequence b).
 * out: [rows][num_heads][head_dim] fp64 (not rounded).  Returns error bits. */
static int32_t run_attention(attn_job* J, int32_t nthreads);

int32_t oracle_paged_attention(
    double* out, const uint16_t* q, int64_t q_row_stride,
    const int32_t* cu_seqlens_q, int32_t num_seqs, const uint16_t* k_cache,
    const uint16_t* v_cache, int32_t num_blocks, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, double scale,
    int32_t partition_tokens, int32_t nthreads) {
  if (num_kv_heads <= 0 || num_heads % num_kv_heads) return -1;
  attn_job J;
  memset(&J, 0, sizeof J);
  J.out = out;
  J.q = q;
  J.q_row_stride = q_row_stride;
  J.cu_seqlens_q = cu_seqlens_q;
  J.num_seqs = num_seqs;
  J.k_cache = k_cache;
  J.v_cache = v_cache;
  J.num_blocks = num_blocks;
  J.block_tables = block_tables;
  J.max_blocks_per_seq = max_blocks_per_seq;
  J.context_lens = context_lens;
  J.num_heads = num_heads;
  J.num_kv_heads = num_kv_heads;
  J.head_dim = head_dim;
  J.block_size = block_size;
  J.scale = scale;
  J.partition_tokens = partition_tokens;
  return run_attention(&J, nthreads);
}

/* The same over an FP8 (e4m3fn) cache: key and value elements are
 * code * k_scale and code * v_scale. */
int32_t oracle_paged_attention_fp8(
    double* out, const uint16_t* q, int64_t q_row_stride,
    const int32_t* cu_seqlens_q, int32_t num_seqs, const uint8_t* k_cache,
    const uint8_t* v_cache, double k_scale, double v_scale, int32_t num_blocks,
    const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, int32_t num_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, double scale, int32_t partition_tokens,
    int32_t nthreads) {
  if (num_kv_heads <= 0 || num_heads % num_kv_heads) return -1;
  attn_job J;
  memset(&J, 0, sizeof J);
  J.out = out;
  J.q = q;
  J.q_row_stride = q_row_stride;
  J.cu_seqlens_q = cu_seqlens_q;
  J.num_seqs = num_seqs;
  J.k_cache8 = k_cache;
  J.v_cache8 = v_cache;
  J.k_scale = k_scale;
  J.v_scale = v_scale;
  J.num_blocks = num_blocks;
  J.block_tables = block_tables;
  J.max_blocks_per_seq = max_blocks_per_seq;
  J.context_lens = context_lens;
  J.num_heads = num_heads;
  J.num_kv_heads = num_kv_heads;
  J.head_dim = head_dim;
  J.block_size = block_size;
  J.scale = scale;
  J.partition_tokens = partition_tokens;
  return run_attention(&J, nthreads);
}

/* Runs the (sequence, head) units of a job over nthreads threads. */
static int32_t run_attention(attn_job* Jp, int32_t nthreads) {
  attn_job J = *Jp;
  pthread_mutex_init(&J.lock, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int32_t started = 0;
  for (int32_t i = 1; i < nthreads; ++i)
    if (pthread_create(&th[started], NULL, attn_worker, &J) == 0) ++started;
  attn_worker(&J);
  for (int32_t i = 0; i < started; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&J.lock);
  return J.err;
}

/* Plain attention over contiguous K/V ([L][Hkv][D], no paging), for the
 * paged-versus-contiguous check.  q: [q_len][H][D]; the q_len queries are
 * the last q_len positions (bottom-right causal).  out fp64 like above. */
int32_t oracle_contiguous_attention(double* out, const uint16_t* q,
                                    const uint16_t* k, const uint16_t* v,
                                    int32_t L, int32_t q_len, int32_t num_heads,
                                    int32_t num_kv_heads, int32_t head_dim,
                                    double scale) {
  if (L <= 0 || q_len <= 0 || q_len > L || num_heads % num_kv_heads) return -1;
  const int32_t D = head_dim, group = num_heads / num_kv_heads;
  double* z = (double*)malloc(sizeof(double) * (size_t)L);
  for (int32_t i = 0; i < q_len; ++i) {
    int32_t last = L - q_len + i;
    for (int32_t h = 0; h < num_heads; ++h) {
      int32_t g = h / group;
      const uint16_t* qh = q + ((int64_t)i * num_heads + h) * D;
      double mx = -INFINITY;
      for (int32_t j = 0; j <= last; ++j) {
        const uint16_t* kj = k + ((int64_t)j * num_kv_heads + g) * D;
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += bf16_to_f64(qh[d]) * bf16_to_f64(kj[d]);
        z[j] = scale * dot;
        mx = z[j] > mx ? z[j] : mx;
      }
      double sum = 0.0;
      double* o = out + ((int64_t)i * num_heads + h) * D;
      for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
      for (int32_t j = 0; j <= last; ++j) {
        double p = exp(z[j] - mx);
        sum += p;
        const uint16_t* vj = v + ((int64_t)j * num_kv_heads + g) * D;
        for (int32_t d = 0; d < D; ++d) o[d] += p * bf16_to_f64(vj[d]);
      }
      for (int32_t d = 0; d < D; ++d) o[d] /= sum;
    }
  }
  free(z);
  return 0;
}
