/*
 * fp8pa_oracle.c -- the CPU oracle for FP8-quantised paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the bench's CPU-baseline leg
 * do.  It shares no code, header, table or constant generator with the CUDA
 * library: every format rule below is written out again from the source
 * pages, on purpose, so that the two sides can disagree.
 *
 * It is plain and slow by design: FP8 decode/encode by explicit bit fields,
 * IEEE fp32 scale arithmetic exactly as the append step defines it, and
 * attention in FP64 with a two-pass softmax over the dequantised cache.
 *
 * Sources (the pages that define the method):
 *  [P1] "DeepSeek V4 950: whole-network FP8 dataflow" (2kiu.com/news/4508674)
 *       sec. 2.1 (E4M3 vs E5M2 roles), sec. 2.2 (MLA latent cache, one scale
 *       per latent group), sec. 2.3 (softmax and accumulators kept in FP32).
 *  [P2] "Llama 3 70B FP8 deployment, 8K-128K long-context tests"
 *       (dpshk.com/news/5605006) sec. 1.1 (E4M3 max 448, smallest non-zero
 *       2^-9), sec. 1.2 (GQA, 64 query heads share 8 KV heads), sec. 3.1
 *       (absmax / 448 scale clamped at 1e-12, then x / scale cast to FP8).
 *  [P4] "FP8混合精度推理全链路部署实战：从模型格式到生产级推理引擎"
 *       (ybb.press/ai-applications/14145.html) sec. 1.1 (E4M3 +-448,
 *       E5M2 +-57344), sec. 2.3 (KV-cache scale management).
 *  [P5] "DeepSeek-V4.1 512K long-context TTFT on 8xH20"
 *       (hotelren.com/news/5711065) sec. 2.2 (blockwise attention with
 *       online softmax), sec. 3.3 (paged KV: fixed-size blocks, one block
 *       table per request).
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes): E4M3 is the "fn" variant (max 448 implies no infinity; S.1111.111
 * is NaN); encode rounds to nearest, ties to even, and saturates finite
 * overflow to +-max; the scale is fp32 absmax / FMAX with IEEE division,
 * clamped below at 1e-12, and codes are fp32 x / scale (a division, not a
 * multiply by the reciprocal); query head h reads KV head h / (Hq / Hkv).
 *
 * The block-scaled mode follows the Microscaling (MX) format that [P4]
 * sec. 7.1 names for Blackwell's FP8 (the page gives only "per-16-element
 * block scaling"): every block of 16 or 32 values along the head dimension
 * shares one power-of-two scale X = 2^e, stored as its biased exponent
 * byte e + 127 (E8M0), with e = floor(log2(block absmax)) - emax, emax the
 * exponent of the format's largest normal (8 for E4M3, 15 for E5M2), held in
 * [-127, 127] (an all-zero block takes e = -127); codes are the FP8 rounding
 * of x / X, saturated.
 *
 * The segment mode is the block-wise cumulative rescaling of [P1] sec. 4.3:
 * the cache is cut into length blocks of 1024 tokens, each block keeps a
 * cumulative scale, and decode dequantises with the scale of the token's
 * block.  The page gives no formula; the reading taken here is the plainest
 * causal one.  Per (sequence, K or V, KV head) a running absmax R covers
 * every token appended so far (it restarts at the sequence's position 0).
 * When the token at position p is appended, R = max(R, absmax of its row);
 * if p is a multiple of 1024 (the token opens segment p / 1024), that
 * segment's scale is frozen as S = max(R / FMAX, 1e-12) (IEEE fp32
 * division), so it is cumulative over all earlier segments and the opening
 * token.  Every token of the segment is coded as x / S; values beyond S *
 * FMAX saturate until the next segment raises S.  Since 1024 is a multiple
 * of every supported block size, each page lies in one segment and stores
 * S once per (page, KV head).
 *
 * The INT8 codec is the alternate KV format the pages mention only as a
 * serving option ("--kv_cache_dtype int8", hotelren.com/news/5166672, the
 * section on inference-engine settings), with no scale or rounding rule.
 * Reading: symmetric codes with FMAX = 127 in place of the FP8 maximum, so
 * the scale is fp32 absmax / 127 (IEEE division, clamped at 1e-12) and the
 * code is x / scale rounded to the nearest integer, ties to even, clamped
 * to [-127, 127], stored as the byte integer + 128 (excess-128: bytes 1 ..
 * 255, 128 for zero); a code's value is its integer, byte - 128.  The
 * power-of-two block mode is defined for FP8 only.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_E4M3 0
#define OR_E5M2 1
#define OR_INT8 2

#define OR_SCALE_TOKEN_HEAD 0
#define OR_SCALE_CHANNEL_STATIC 1
#define OR_SCALE_TOKEN_GROUP 2
#define OR_SCALE_MX_BLOCK 3
#define OR_SCALE_SEGMENT 4

/* Tokens per segment of the block-wise cumulative rescaling ([P1] sec. 4.3:
 * the extra offset is refreshed every 1024 tokens). */
#define OR_SEGMENT_TOKENS 1024

/* ------------------------------------------------------------------ */
/* FP8 formats: [P2] sec. 1.1, [P4] sec. 1.1, [P1] sec. 2.1.           */
/* ------------------------------------------------------------------ */

/* Largest finite magnitude: 448 for E4M3, 57344 for E5M2 ([P4] sec. 1.1),
 * 127 for the symmetric INT8 codec. */
double or_fp8_max(int fmt) {
  return fmt == OR_E4M3 ? 448.0 : (fmt == OR_E5M2 ? 57344.0 : 127.0);
}

/* Value of an FP8 code, read field by field.
 * E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent field 0 is
 *       subnormal (m/8)*2^-6; S.1111.111 is NaN; there is no infinity.
 * E5M2: 1 sign, 5 exponent (bias 15), 2 mantissa bits; exponent field 0 is
 *       subnormal (m/4)*2^-14; exponent field 31 is inf (m = 0) or NaN. */
double or_fp8_decode(uint8_t code, int fmt) {
  if (fmt == OR_INT8) return (double)((int)code - 128);
  int neg = (code >> 7) & 1;
  double mag;
  if (fmt == OR_E4M3) {
    int e = (code >> 3) & 0xF, m = code & 0x7;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
      mag = ldexp((double)m / 8.0, -6);
    else
      mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  } else {
    int e = (code >> 2) & 0x1F, m = code & 0x3;
    if (e == 0x1F) {
      if (m != 0) return NAN;
      mag = INFINITY;
    } else if (e == 0) {
      mag = ldexp((double)m / 4.0, -14);
    } else {
      mag = ldexp(1.0 + (double)m / 4.0, e - 15);
    }
  }
  return neg ? -mag : mag;
}

/* fp32 -> INT8 code: the nearest integer (from the floor and the remainder),
 * ties to the even one, clamped to [-127, 127], NaN -> 0; stored + 128. */
static uint8_t or_int8_encode(float x) {
  if (isnan(x)) return 128;
  const double xd = (double)x;
  if (xd >= 127.0) return 127 + 128;
  if (xd <= -127.0) return -127 + 128;
  const double f = floor(xd);
  const double r = xd - f; /* exact: |xd| < 2^7 */
  long n = (long)f;
  if (r > 0.5 || (r == 0.5 && (n & 1l))) n += 1;
  return (uint8_t)(n + 128);
}

/* fp32 -> FP8 code by integer manipulation of the fp32 bit pattern:
 * round to nearest, ties to even, saturate finite overflow (and +-inf) to
 * +-max, keep the sign of zero, NaN -> 0x7F.  (INT8: or_int8_encode.) */
uint8_t or_fp8_encode(float x, int fmt) {
  if (fmt == OR_INT8) return or_int8_encode(x);
  uint32_t bits;
  memcpy(&bits, &x, sizeof bits);
  const uint32_t sign = (bits >> 31) ? 0x80u : 0x00u;
  const uint32_t fexp = (bits >> 23) & 0xFFu;
  const uint32_t fman = bits & 0x7FFFFFu;
  const int mbits = (fmt == OR_E4M3) ? 3 : 2;     /* stored mantissa bits */
  const int bias = (fmt == OR_E4M3) ? 7 : 15;     /* exponent bias        */
  const int emin = 1 - bias;                      /* smallest normal exp  */
  const int maxcode = (fmt == OR_E4M3) ? 0x7E : 0x7B; /* +max magnitude  */

  if (fexp == 0xFFu) return fman ? 0x7F : (uint8_t)(sign | (uint32_t)maxcode);
  /* fp32 zeros and subnormals are below 2^-126: far under half of the
   * smallest FP8 subnormal, so they round to a signed zero. */
  if (fexp == 0u) return (uint8_t)sign;

  const int e = (int)fexp - 127;                  /* x = sig * 2^(e-23)  */
  const uint64_t sig = (uint64_t)(0x800000u | fman);
  /* The target grid spacing is 2^(max(e, emin) - mbits). */
  const int q = (e >= emin ? e : emin) - mbits;
  const int sh = q - (e - 23);                    /* >= 23 - mbits > 0   */
  uint64_t n;
  if (sh >= 40) {
    n = 0;                                        /* far below half step */
  } else {
    n = sig >> sh;
    const uint64_t rem = sig & ((1ull << sh) - 1ull);
    const uint64_t half = 1ull << (sh - 1);
    if (rem > half || (rem == half && (n & 1ull))) n += 1;
  }
  long code;
  if (e >= emin) {
    /* n in [2^mbits, 2^(mbits+1)]; n == 2^(mbits+1) carries into the
     * exponent field by the plain addition below. */
    code = ((long)(e + bias) << mbits) + (long)n - (1l << mbits);
  } else {
    code = (long)n; /* subnormal: n in [0, 2^mbits]; 2^mbits = min normal */
  }
  if (code > maxcode) code = maxcode;             /* satfinite           */
  return (uint8_t)(sign | (uint32_t)code);
}

/* A second, independent encoder used only to pin the first: scan all codes
 * of the same sign for the nearest value in FP64; ties go to the code with
 * an even mantissa (an even code number); beyond max it saturates. */
uint8_t or_fp8_encode_bruteforce(float x, int fmt) {
  if (fmt == OR_INT8) {
    /* beyond the range it clamps; inside, scan every integer in
     * [-127, 127] for the nearest, ties to the even one */
    if (isnan(x)) return 128;
    if ((double)x >= 127.0) return 127 + 128;
    if ((double)x <= -127.0) return -127 + 128;
    int best = 0;
    double bestd = INFINITY;
    for (int c = -127; c <= 127; ++c) {
      const double d = fabs((double)c - (double)x);
      if (d < bestd || (d == bestd && (c & 1) == 0)) {
        bestd = d;
        best = c;
      }
    }
    return (uint8_t)(best + 128);
  }
  if (isnan(x)) return 0x7F;
  const double xd = (double)x;
  const int neg = signbit(x) ? 1 : 0;
  const double fmax = or_fp8_max(fmt);
  if (fabs(xd) >= fmax) return (uint8_t)((neg ? 0x80 : 0) | (fmt == OR_E4M3 ? 0x7E : 0x7B));
  int best = -1;
  double bestd = INFINITY;
  for (int c = 0; c < 128; ++c) {
    const int code = (neg ? 0x80 : 0) | c;
    const double v = or_fp8_decode((uint8_t)code, fmt);
    if (!isfinite(v)) continue;
    const double d = fabs(v - xd);
    if (d < bestd || (d == bestd && (code & 1) == 0 && (best & 1) == 1)) {
      bestd = d;
      best = code;
    }
  }
  return (uint8_t)best;
}

void or_fp8_encode_array(const float* x, long n, int fmt, uint8_t* out) {
  for (long i = 0; i < n; ++i) out[i] = or_fp8_encode(x[i], fmt);
}
void or_fp8_encode_bruteforce_array(const float* x, long n, int fmt, uint8_t* out) {
  for (long i = 0; i < n; ++i) out[i] = or_fp8_encode_bruteforce(x[i], fmt);
}
void or_fp8_decode_array(const uint8_t* c, long n, int fmt, double* out) {
  for (long i = 0; i < n; ++i) out[i] = or_fp8_decode(c[i], fmt);
}

/* ------------------------------------------------------------------ */
/* Append: absmax scale, quantise, scatter ([P2] sec. 3.1, [P4] sec.   */
/* 2.3, [P1] sec. 2.2 / 2.4, [P5] sec. 3.3).                           */
/* ------------------------------------------------------------------ */

static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* The absmax scale of one group of values: fp32 absmax / FMAX with IEEE
 * fp32 division, clamped below at 1e-12 ([P2] sec. 3.1). */
static float or_absmax_scale(const float* x, int n, int fmt) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) amax = fmaxf(amax, fabsf(x[i]));
  volatile float fmax_f = (float)or_fp8_max(fmt);
  float s = amax / fmax_f;
  return fmaxf(s, 1e-12f);
}

float or_absmax_scale_bf16(const uint16_t* x, int n, int fmt) {
  float* tmp = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
  for (int i = 0; i < n; ++i) tmp[i] = bf16_to_f32(x[i]);
  float s = or_absmax_scale(tmp, n, fmt);
  free(tmp);
  return s;
}

/* The block exponent e of the MX mode: floor(log2(amax)) - emax, in
 * [-127, 127]; -127 for amax = 0.  frexp gives amax = m * 2^E, m in
 * [0.5, 1), so floor(log2(amax)) = E - 1 exactly. */
int or_mx_exponent(float amax, int fmt) {
  if (!(amax > 0.0f)) return -127;
  int E = 0;
  (void)frexp((double)amax, &E);
  int e = (E - 1) - (fmt == OR_E4M3 ? 8 : 15);
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

/* Quantise one row of `d` values and store codes (and scales) in the
 * paged layout:
 *   codes  [num_blocks][Hkv][bs][D]        u8
 *   TOKEN_HEAD  scale [num_blocks][Hkv][bs]           f32 (written)
 *   TOKEN_GROUP scale [num_blocks][Hkv][bs][D / gs]   f32 (written)
 *   CHANNEL_STATIC scale [Hkv][D]                     f32 (read)
 *   MX_BLOCK scale [num_blocks][Hkv][bs][D / gs]      u8 E8M0 (written) */
static void or_quant_row(const uint16_t* src, int d, int fmt, int mode, int gs,
                         const float* chan_scale, uint8_t* dst_codes,
                         void* dst_scale) {
  float* x = (float*)malloc(sizeof(float) * (size_t)d);
  for (int i = 0; i < d; ++i) x[i] = bf16_to_f32(src[i]);
  if (mode == OR_SCALE_TOKEN_HEAD) {
    const float s = or_absmax_scale(x, d, fmt);
    for (int i = 0; i < d; ++i) dst_codes[i] = or_fp8_encode(x[i] / s, fmt);
    *(float*)dst_scale = s;
  } else if (mode == OR_SCALE_TOKEN_GROUP) {
    for (int g = 0; g < d / gs; ++g) {
      const float s = or_absmax_scale(x + g * gs, gs, fmt);
      for (int i = 0; i < gs; ++i)
        dst_codes[g * gs + i] = or_fp8_encode(x[g * gs + i] / s, fmt);
      ((float*)dst_scale)[g] = s;
    }
  } else if (mode == OR_SCALE_MX_BLOCK) {
    for (int g = 0; g < d / gs; ++g) {
      float amax = 0.0f;
      for (int i = 0; i < gs; ++i) amax = fmaxf(amax, fabsf(x[g * gs + i]));
      const int e = or_mx_exponent(amax, fmt);
      /* x / 2^e is exact in FP64; the float conversion rounds only below
       * the fp32 normal range, where every such value encodes to zero. */
      for (int i = 0; i < gs; ++i)
        dst_codes[g * gs + i] = or_fp8_encode((float)ldexp((double)x[g * gs + i], -e), fmt);
      ((uint8_t*)dst_scale)[g] = (uint8_t)(e + 127);
    }
  } else {
    for (int i = 0; i < d; ++i) dst_codes[i] = or_fp8_encode(x[i] / chan_scale[i], fmt);
  }
  free(x);
}

/* k, v: bf16 [num_tokens][Hkv][D]; v may be NULL (one shared latent).
 * slot_mapping[t] < 0 skips token t; a slot past the pool is skipped and
 * counted.  Returns the number of skipped out-of-range slots. */
int or_kv_append_quant(const uint16_t* k, const uint16_t* v, const int32_t* slot_mapping,
                       int num_tokens, int n_kv_heads, int head_dim, int fmt, int scale_mode,
                       int group_size, uint8_t* k_cache, uint8_t* v_cache, float* k_scale,
                       float* v_scale, int num_blocks, int block_size) {
  int bad = 0;
  const int ngroups = (scale_mode == OR_SCALE_TOKEN_GROUP || scale_mode == OR_SCALE_MX_BLOCK)
                          ? head_dim / group_size
                          : 1;
  for (int t = 0; t < num_tokens; ++t) {
    const int slot = slot_mapping[t];
    if (slot < 0) continue;
    const long blk = slot / block_size, off = slot % block_size;
    if (blk >= num_blocks) {
      ++bad;
      continue;
    }
    for (int h = 0; h < n_kv_heads; ++h) {
      const long row = (blk * n_kv_heads + h) * block_size + off;
      for (int which = 0; which < 2; ++which) {
        const uint16_t* src = which == 0 ? k : v;
        if (src == NULL) continue;
        uint8_t* cache = which == 0 ? k_cache : v_cache;
        float* sc = which == 0 ? k_scale : v_scale;
        const uint16_t* x = src + ((long)t * n_kv_heads + h) * head_dim;
        void* dst_scale = NULL;
        const float* chan = NULL;
        if (scale_mode == OR_SCALE_CHANNEL_STATIC)
          chan = sc + (long)h * head_dim;
        else if (scale_mode == OR_SCALE_MX_BLOCK)
          dst_scale = (uint8_t*)sc + row * ngroups;  /* E8M0 bytes */
        else
          dst_scale = sc + row * ngroups;
        or_quant_row(x, head_dim, fmt, scale_mode, group_size, chan, cache + row * head_dim,
                     dst_scale);
      }
    }
  }
  return bad;
}

/* Static per-channel scales for CHANNEL_STATIC mode: for every (kv_head,
 * dim) the absmax over all tokens, / FMAX, clamped at 1e-12.
 * x: bf16 [num_tokens][Hkv][D]; out: f32 [Hkv][D]. */
void or_kv_channel_scales(const uint16_t* x, int num_tokens, int n_kv_heads, int head_dim,
                          int fmt, float* out) {
  const long n = (long)n_kv_heads * head_dim;
  float* amax = (float*)calloc((size_t)n, sizeof(float));
  for (long t = 0; t < num_tokens; ++t)
    for (long i = 0; i < n; ++i) amax[i] = fmaxf(amax[i], fabsf(bf16_to_f32(x[t * n + i])));
  volatile float fmax_f = (float)or_fp8_max(fmt);
  for (long i = 0; i < n; ++i) out[i] = fmaxf(amax[i] / fmax_f, 1e-12f);
  free(amax);
}

/* Heads per page row of the segment scale array: n_kv_heads rounded up to a
 * multiple of 4 (one 16-byte row per page). */
static int or_seg_heads(int n_kv_heads) { return (n_kv_heads + 3) / 4 * 4; }

/* Segment-scale append ([P1] sec. 4.3, read as in the header above).
 * k, v: bf16 [num_tokens][Hkv][D] (v may be NULL); the tokens of sequence r
 * are rows seq_offsets[r] .. seq_offsets[r+1]-1, at positions
 * seq_start_pos[r], +1, ...  seg_state f32 [num_seqs][2][Hkv][2] carries
 * (R, S) of every (sequence, K or V, head) between calls.  Scales:
 * f32 [num_blocks][round_up(Hkv, 4)], the segment scale of each page.
 * A token whose slot is negative or past the pool is skipped (it neither
 * raises R nor opens its segment).  Returns the count of out-of-range
 * slots. */
int or_kv_append_quant_segment(const uint16_t* k, const uint16_t* v,
                               const int32_t* slot_mapping, const int32_t* seq_offsets,
                               const int32_t* seq_start_pos, int num_seqs, int n_kv_heads,
                               int head_dim, int fmt, float* seg_state, uint8_t* k_cache,
                               uint8_t* v_cache, float* k_scale, float* v_scale, int num_blocks,
                               int block_size) {
  int bad = 0;
  const int hp = or_seg_heads(n_kv_heads);
  volatile float fmax_f = (float)or_fp8_max(fmt);
  float* x = (float*)malloc(sizeof(float) * (size_t)head_dim);
  for (int r = 0; r < num_seqs; ++r) {
    for (int which = 0; which < 2; ++which) {
      const uint16_t* src = which == 0 ? k : v;
      if (src == NULL) continue;
      uint8_t* cache = which == 0 ? k_cache : v_cache;
      float* sc = which == 0 ? k_scale : v_scale;
      for (int h = 0; h < n_kv_heads; ++h) {
        float* st = seg_state + (((long)r * 2 + which) * n_kv_heads + h) * 2;
        float R = st[0], S = st[1];
        for (int i = seq_offsets[r]; i < seq_offsets[r + 1]; ++i) {
          const long p = (long)seq_start_pos[r] + (i - seq_offsets[r]);
          if (p == 0) R = 0.0f; /* a new sequence */
          const int slot = slot_mapping[i];
          if (slot < 0) continue;
          const long blk = slot / block_size, off = slot % block_size;
          if (blk >= num_blocks) {
            if (which == 0 && h == 0) ++bad;
            continue;
          }
          const uint16_t* row = src + ((long)i * n_kv_heads + h) * head_dim;
          float amax = 0.0f;
          for (int d = 0; d < head_dim; ++d) {
            x[d] = bf16_to_f32(row[d]);
            amax = fmaxf(amax, fabsf(x[d]));
          }
          R = fmaxf(R, amax);
          if (p % OR_SEGMENT_TOKENS == 0) S = fmaxf(R / fmax_f, 1e-12f);
          uint8_t* dst = cache + (((long)blk * n_kv_heads + h) * block_size + off) * head_dim;
          for (int d = 0; d < head_dim; ++d) dst[d] = or_fp8_encode(x[d] / S, fmt);
          sc[blk * hp + h] = S;
        }
        st[0] = R;
        st[1] = S;
      }
    }
  }
  free(x);
  return bad;
}

/* ------------------------------------------------------------------ */
/* Attention over the paged, dequantised cache in FP64                */
/* ([P2] sec. 1.2 GQA, [P1] sec. 2.3 softmax, [P5] sec. 2.2 / 3.3).    */
/* ------------------------------------------------------------------ */

typedef struct {
  const uint16_t* q;            /* bf16 [B][Hq][Dk]                    */
  const uint8_t* k_cache;       /* [nb][Hkv][bs][Dk]                   */
  const uint8_t* v_cache;       /* [nb][Hkv][bs][Dk]; may be k_cache   */
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_tables;  /* [B][max_blocks]                     */
  int max_blocks;
  const int32_t* seq_lens;      /* [B]                                 */
  int batch, block_size, hq, hkv, dk, dv, fmt, mode, gs, num_blocks;
  double sm_scale;
} or_attn_t;

/* Dequantised element d of token t of request b, kv head g, from `cache`
 * with scales `sc`: decode(code) * scale, both read into FP64.  Returns 0
 * and sets *ok = 0 on an out-of-range block id. */
static double or_deq(const or_attn_t* a, const uint8_t* cache, const float* sc, int b, int g,
                     int t, int d, int* ok) {
  const int blk = a->block_tables[(long)b * a->max_blocks + t / a->block_size];
  const int off = t % a->block_size;
  if (blk < 0 || blk >= a->num_blocks) {
    *ok = 0;
    return 0.0;
  }
  const long row = ((long)blk * a->hkv + g) * a->block_size + off;
  const double code = or_fp8_decode(cache[row * a->dk + d], a->fmt);
  double s;
  if (a->mode == OR_SCALE_TOKEN_HEAD)
    s = (double)sc[row];
  else if (a->mode == OR_SCALE_TOKEN_GROUP)
    s = (double)sc[row * (a->dk / a->gs) + d / a->gs];
  else if (a->mode == OR_SCALE_MX_BLOCK)
    s = ldexp(1.0, (int)((const uint8_t*)sc)[row * (a->dk / a->gs) + d / a->gs] - 127);
  else if (a->mode == OR_SCALE_SEGMENT)
    s = (double)sc[(long)blk * or_seg_heads(a->hkv) + g];
  else
    s = (double)sc[(long)g * a->dk + d];
  return code * s;
}

/* Scores z_t = sm_scale * sum_d q_d * k^_{t,d} for one (b, h) row. */
static void or_scores(const or_attn_t* a, int b, int h, int L, double* z, int* ok) {
  const int g = h / (a->hq / a->hkv);
  const uint16_t* q = a->q + ((long)b * a->hq + h) * a->dk;
  for (int t = 0; t < L; ++t) {
    double acc = 0.0;
    for (int d = 0; d < a->dk; ++d)
      acc += (double)bf16_to_f32(q[d]) * or_deq(a, a->k_cache, a->k_scale, b, g, t, d, ok);
    z[t] = a->sm_scale * acc;
  }
}

/* One output row, two-pass softmax: m = max z, p = exp(z - m), l = sum p,
 * o = sum p v^ / l.  L = 0 gives a zero row. */
static void or_attn_row(const or_attn_t* a, int b, int h, double* out, double* z, int* ok) {
  int L = a->seq_lens[b];
  if (L > a->max_blocks * a->block_size) L = a->max_blocks * a->block_size;
  for (int d = 0; d < a->dv; ++d) out[d] = 0.0;
  if (L <= 0) return;
  const int g = h / (a->hq / a->hkv);
  or_scores(a, b, h, L, z, ok);
  double m = -INFINITY;
  for (int t = 0; t < L; ++t) m = z[t] > m ? z[t] : m;
  double l = 0.0;
  for (int t = 0; t < L; ++t) {
    z[t] = exp(z[t] - m);
    l += z[t];
  }
  for (int t = 0; t < L; ++t) {
    const double p = z[t] / l;
    for (int d = 0; d < a->dv; ++d) out[d] += p * or_deq(a, a->v_cache, a->v_scale, b, g, t, d, ok);
  }
}

/* Full or sampled attention.  rows == NULL computes every (b, h) row into
 * out [B][Hq][Dv]; otherwise rows[i] = b * Hq + h and out is [n_rows][Dv].
 * Rows run in parallel on `num_threads` host threads.  Returns the number
 * of rows that met an out-of-range block id. */
int or_paged_decode_attention(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                              const float* k_scale, const float* v_scale,
                              const int32_t* block_tables, int max_blocks_per_seq,
                              const int32_t* seq_lens, int batch, int block_size, int n_q_heads,
                              int n_kv_heads, int head_dim, int head_dim_v, int fmt,
                              int scale_mode, int group_size, double sm_scale, int num_blocks,
                              const int32_t* rows, int n_rows, double* out, int num_threads) {
  or_attn_t a = {q,        k_cache,    v_cache,  k_scale,   v_scale,    block_tables,
                 max_blocks_per_seq,   seq_lens, batch,     block_size, n_q_heads,
                 n_kv_heads, head_dim, head_dim_v, fmt,     scale_mode, group_size,
                 num_blocks, sm_scale};
  const int total = rows ? n_rows : batch * n_q_heads;
  int bad = 0;
  if (num_threads < 1) num_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(+ : bad)
  for (int i = 0; i < total; ++i) {
    const int r = rows ? rows[i] : i;
    const int b = r / n_q_heads, h = r % n_q_heads;
    int ok = 1;
    double* z = (double*)malloc(sizeof(double) * (size_t)(max_blocks_per_seq * block_size + 1));
    or_attn_row(&a, b, h, out + (long)i * head_dim_v, z, &ok);
    free(z);
    if (!ok) ++bad;
  }
  return bad;
}

/* The normalised softmax weights p_t / l of one (b, h) row (for the
 * "weights sum to one" check).  Returns L. */
int or_attention_weights(const uint16_t* q, const uint8_t* k_cache, const float* k_scale,
                         const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* seq_lens, int block_size, int n_q_heads, int n_kv_heads,
                         int head_dim, int fmt, int scale_mode, int group_size, double sm_scale,
                         int num_blocks, int b, int h, double* w) {
  or_attn_t a = {q,        k_cache,    k_cache,  k_scale,  k_scale,    block_tables,
                 max_blocks_per_seq,   seq_lens, b + 1,    block_size, n_q_heads,
                 n_kv_heads, head_dim, head_dim, fmt,      scale_mode, group_size,
                 num_blocks, sm_scale};
  const int L = seq_lens[b];
  int ok = 1;
  if (L <= 0) return 0;
  or_scores(&a, b, h, L, w, &ok);
  double m = -INFINITY, l = 0.0;
  for (int t = 0; t < L; ++t) m = w[t] > m ? w[t] : m;
  for (int t = 0; t < L; ++t) {
    w[t] = exp(w[t] - m);
    l += w[t];
  }
  for (int t = 0; t < L; ++t) w[t] /= l;
  return L;
}

/* The same attention written as independent token chunks, each giving a
 * partial (m_i, l_i, o_i) with o_i unnormalised, merged by
 * M = max m_i, l = sum e^(m_i - M) l_i, o = sum e^(m_i - M) o_i / l.
 * It exists to pin the split-K merge algebra against the two-pass form. */
void or_attention_split_merge(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                              const float* k_scale, const float* v_scale,
                              const int32_t* block_tables, int max_blocks_per_seq,
                              const int32_t* seq_lens, int batch, int block_size, int n_q_heads,
                              int n_kv_heads, int head_dim, int head_dim_v, int fmt,
                              int scale_mode, int group_size, double sm_scale, int num_blocks,
                              int chunk_tokens, double* out) {
  or_attn_t a = {q,        k_cache,    v_cache,  k_scale,   v_scale,    block_tables,
                 max_blocks_per_seq,   seq_lens, batch,     block_size, n_q_heads,
                 n_kv_heads, head_dim, head_dim_v, fmt,     scale_mode, group_size,
                 num_blocks, sm_scale};
  const int dv = head_dim_v;
  double* z = (double*)malloc(sizeof(double) * (size_t)(max_blocks_per_seq * block_size + 1));
  double* oi = (double*)malloc(sizeof(double) * (size_t)dv);
  for (int b = 0; b < batch; ++b) {
    for (int h = 0; h < n_q_heads; ++h) {
      double* o = out + ((long)b * n_q_heads + h) * dv;
      for (int d = 0; d < dv; ++d) o[d] = 0.0;
      const int L = seq_lens[b];
      if (L <= 0) continue;
      const int g = h / (n_q_heads / n_kv_heads);
      int ok = 1;
      or_scores(&a, b, h, L, z, &ok);
      double M = -INFINITY, lsum = 0.0;
      for (int t0 = 0; t0 < L; t0 += chunk_tokens) {
        const int t1 = t0 + chunk_tokens < L ? t0 + chunk_tokens : L;
        double mi = -INFINITY, li = 0.0;
        for (int t = t0; t < t1; ++t) mi = z[t] > mi ? z[t] : mi;
        for (int d = 0; d < dv; ++d) oi[d] = 0.0;
        for (int t = t0; t < t1; ++t) {
          const double p = exp(z[t] - mi);
          li += p;
          for (int d = 0; d < dv; ++d) oi[d] += p * or_deq(&a, v_cache, v_scale, b, g, t, d, &ok);
        }
        /* merge the running state (M, lsum, o) with (mi, li, oi) */
        const double Mn = mi > M ? mi : M;
        const double wa = (M == -INFINITY) ? 0.0 : exp(M - Mn);
        const double wb = exp(mi - Mn);
        for (int d = 0; d < dv; ++d) o[d] = o[d] * wa + oi[d] * wb;
        lsum = lsum * wa + li * wb;
        M = Mn;
      }
      for (int d = 0; d < dv; ++d) o[d] /= lsum;
    }
  }
  free(z);
  free(oi);
}

int or_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
