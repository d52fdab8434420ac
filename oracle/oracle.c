/*
 * Float64 CPU oracle for the tiled / top-k / sparse attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously correct
 * reference the CUDA path is checked against. Only the test-suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the product path
 * never calls it. It shares no code, header, table or helper with the CUDA
 * library.
 *
 * Sources ("the pages"):
 *   [p1] "DeepSeek V4.1 上 4×RTX 3090：视觉链路的两个坑和修复" (blog.erguotou.me),
 *        section 三 (piece-wise attention: S = Q_blk K^T, row softmax, P V, rows
 *        mapped back to q0..q0+qb) and section 四 (softmax rows sum to 1).
 *   [p2] "AMD MI250部署DeepSeek-V4-Flash：先修正确性再谈性能" (yfxerp.com),
 *        sections 3.1 / 4.1 (softmax statistics kept in higher precision),
 *        3.3 (causal mask as -inf), 4.2 (fixed tie-break for top-k).
 *   [p3] "从 SGLang Kernel源码到 GPU Trace：DeepSeek V4.1 Flash - Prefill"
 *        (gsyq.cn), sections 2.2 / 3.2 (variable-length batches described by
 *        cu_seqlens_q / cu_seqlens_k; keys past a sequence's length are skipped).
 *   [p4] "推理引擎的蝴蝶效应 -- 从V32 模型的输出不一致说起" (edward-lyz.github.io),
 *        sections 实验方法和结果 (top-k over indexer logits with row_starts /
 *        row_lens, (323, 2590) -> (323, 2048); gather through pagetable_1;
 *        sorting the index list restores identical output; stable sort as the
 *        top-k fix) and 进一步探索 (equations 1-2, the online-softmax merge).
 *
 * All arithmetic is double precision. Inputs are float arrays holding exactly
 * the values the GPU consumes (bf16 values widen exactly to float).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16 rounding (round to nearest, ties to even) of an fp32 value.          */
/* The GPU path rounds fp32 inputs to bf16 at its boundary; the oracle         */
/* reproduces that input rounding itself (textbook RNE on the top 16 bits).    */
/* NaN/Inf are passed through unchanged (the generators never produce them). */
void oracle_round_bf16(const float* in, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) {
    uint32_t u;
    memcpy(&u, &in[i], 4);
    if ((u & 0x7F800000u) != 0x7F800000u) {
      uint32_t lsb = (u >> 16) & 1u;
      u = (u + 0x7FFFu + lsb) & 0xFFFF0000u;
    }
    memcpy(&out[i], &u, 4);
  }
}

/* ------------------------------------------------------------------------ */
/* O1. Dense attention over packed variable-length sequences.                */
/*                                                                           */
/* q   [total_q, hq,  d]   k, v [total_k, hkv, d]   (d contiguous)           */
/* cu_q, cu_k [batch+1] prefix sums of sequence lengths ([p3] 2.2).          */
/* For sequence b, head h, query row i (0-based within the sequence):        */
/*   g = h / (hq / hkv)                      (grouped KV heads)               */
/*   visible keys j in [0, Lk); causal keeps j <= i + (Lk - Lq)               */
/*   s_j = scale * sum_t q[i,h,t] k[j,g,t]            ([p1] S-gemm)           */
/*   m = max_j s_j;  p_j = exp(s_j - m) / sum_j exp(s_j - m)  ([p1] softmax)  */
/*   out[i,h,:] = sum_j p_j v[j,g,:]                  ([p1] PV-gemm)          */
/*   lse[i,h] = m + ln sum_j exp(s_j - m)                                    */
/* A row with no visible key gets out = 0 and lse = -inf.                    */
/*                                                                           */
/* rows == NULL: every (token, head) row. Otherwise only the n_rows rows      */
/* (tok[r], head[r]); results go to out[r*d..], lse[r].                      */
/* Returns 0, or -1 when cu_q / cu_k are not non-decreasing from 0.          */
static int find_seq(const int32_t* cu, int batch, int32_t tok) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) { /* last b with cu[b] <= tok */
    int mid = (lo + hi + 1) / 2;
    if (cu[mid] <= tok) lo = mid; else hi = mid - 1;
  }
  return lo;
}

static void attn_row(const float* q, const float* k, const float* v, const int32_t* cu_q,
                     const int32_t* cu_k, int batch, int hq, int hkv, int d, int causal,
                     double scale, int32_t tok, int h, double* out_row, double* lse_row,
                     double* s /* scratch, max_lk */) {
  const int b = find_seq(cu_q, batch, tok);
  const int64_t Lq = cu_q[b + 1] - cu_q[b];
  const int64_t Lk = cu_k[b + 1] - cu_k[b];
  const int64_t i = tok - cu_q[b];
  const int g = h / (hq / hkv);
  int64_t nvis = Lk;
  if (causal) {
    int64_t lim = i + (Lk - Lq) + 1; /* keys 0..i+(Lk-Lq) */
    if (lim < nvis) nvis = lim;
    if (nvis < 0) nvis = 0;
  }
  for (int t = 0; t < d; ++t) out_row[t] = 0.0;
  if (nvis == 0) {
    *lse_row = -INFINITY;
    return;
  }
  const float* qi = q + ((int64_t)tok * hq + h) * d;
  double m = -INFINITY;
  for (int64_t j = 0; j < nvis; ++j) {
    const float* kj = k + ((int64_t)(cu_k[b] + j) * hkv + g) * d;
    double acc = 0.0;
    for (int t = 0; t < d; ++t) acc += (double)qi[t] * (double)kj[t];
    s[j] = scale * acc;
    if (s[j] > m) m = s[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j < nvis; ++j) {
    s[j] = exp(s[j] - m);
    l += s[j];
  }
  for (int64_t j = 0; j < nvis; ++j) {
    const float* vj = v + ((int64_t)(cu_k[b] + j) * hkv + g) * d;
    const double p = s[j] / l;
    for (int t = 0; t < d; ++t) out_row[t] += p * (double)vj[t];
  }
  *lse_row = m + log(l);
}

int oracle_attn_varlen(const float* q, const float* k, const float* v, const int32_t* cu_q,
                       const int32_t* cu_k, int batch, int hq, int hkv, int d, int causal,
                       double scale, const int32_t* tok, const int32_t* head, int64_t n_rows,
                       double* out, double* lse) {
  if (batch < 1 || hq < 1 || hkv < 1 || d < 1 || hq % hkv != 0) return -2;
  if (cu_q[0] != 0 || cu_k[0] != 0) return -1;
  int64_t max_lk = 0;
  for (int b = 0; b < batch; ++b) {
    if (cu_q[b + 1] < cu_q[b] || cu_k[b + 1] < cu_k[b]) return -1;
    if (cu_k[b + 1] - cu_k[b] > max_lk) max_lk = cu_k[b + 1] - cu_k[b];
  }
  const int64_t total_q = cu_q[batch];
  const int64_t n = (tok == NULL) ? total_q * hq : n_rows;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_lk > 0 ? max_lk : 1));
#pragma omp for schedule(dynamic, 16)
    for (int64_t r = 0; r < n; ++r) {
      int32_t t_ = (tok == NULL) ? (int32_t)(r / hq) : tok[r];
      int h_ = (tok == NULL) ? (int)(r % hq) : head[r];
      attn_row(q, k, v, cu_q, cu_k, batch, hq, hkv, d, causal, scale, t_, h_, out + r * d,
               lse + r, s);
    }
    free(s);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* O2. Top-k selection ([p4] 实验方法和结果; [p2] 4.2).                      */
/*                                                                           */
/* Row r's window is logits[r*row_stride + row_starts[r] ..+ row_lens[r]).   */
/* The result is what a stable descending sort gives: positions ordered by   */
/* value descending, equal values by ascending position (lower index wins).  */
/* idx[r, 0:min(k,len)] = the first min(k,len) positions (relative to the    */
/* window start); the remaining slots are -1. A window that does not fit the */
/* row (negative start/len, or start+len > row_stride) gives an all -1 row   */
/* and is counted in the return value. Floats compare as floats: -0 == +0.   */
typedef struct {
  float v;
  int32_t pos;
} vp_t;

static int cmp_desc_stable(const void* a, const void* b) {
  const vp_t* x = (const vp_t*)a;
  const vp_t* y = (const vp_t*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->pos > y->pos) - (x->pos < y->pos);
}

int64_t oracle_topk(const float* logits, int64_t row_stride, int64_t rows,
                    const int32_t* row_starts, const int32_t* row_lens, int k, int32_t* idx) {
  int64_t bad = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(+ : bad)
  for (int64_t r = 0; r < rows; ++r) {
    int32_t* out = idx + r * (int64_t)k;
    for (int j = 0; j < k; ++j) out[j] = -1;
    const int64_t st = row_starts[r], len = row_lens[r];
    if (st < 0 || len < 0 || st + len > row_stride) {
      bad += 1;
      continue;
    }
    vp_t* w = (vp_t*)malloc(sizeof(vp_t) * (size_t)(len > 0 ? len : 1));
    for (int64_t j = 0; j < len; ++j) {
      w[j].v = logits[r * row_stride + st + j];
      w[j].pos = (int32_t)j;
    }
    /* The comparator is a total order, so this equals a stable sort by value. */
    qsort(w, (size_t)len, sizeof(vp_t), cmp_desc_stable);
    const int64_t take = len < k ? len : k;
    for (int64_t j = 0; j < take; ++j) out[j] = w[j].pos;
    free(w);
  }
  return bad;
}

/* ------------------------------------------------------------------------ */
/* O3. Sparse attention through a paged KV cache ([p4] 实验方法和结果,       */
/* 进一步探索).                                                               */
/*                                                                           */
/* q        [nq, H, dqk]                                                     */
/* kv_cache [num_pages, page_size, dqk]; K = a row's dqk values, V = its     */
/*          first dv values (one latent shared by K and V).                  */
/* page_table[num_logical_pages]: logical page -> physical page.             */
/* idx      [nq, topk] logical token positions; -1 = empty slot.             */
/* For query n: drop -1 entries and entries outside [0, kv_len) or whose     */
/* page maps outside [0, num_pages) (counted in the return value); sort the   */
/* rest ascending (the canonical order; duplicates keep their multiplicity);  */
/* gather row = kv_cache[page_table[i / page_size], i % page_size]; then per  */
/* head plain softmax attention with scale, exactly as O1 (one KV head).      */
/* A query with no valid entry gets out = 0, lse = -inf.                     */
static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

int64_t oracle_sparse_paged(const float* q, int64_t nq, int H, int dqk, int dv,
                            const float* kv_cache, int64_t num_pages, int page_size,
                            const int32_t* page_table, int64_t num_logical_pages, int64_t kv_len,
                            const int32_t* idx, int topk, double scale, double* out,
                            double* lse) {
  int64_t bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
  for (int64_t n = 0; n < nq; ++n) {
    int32_t* list = (int32_t*)malloc(sizeof(int32_t) * (size_t)(topk > 0 ? topk : 1));
    double* s = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1));
    int cnt = 0;
    for (int j = 0; j < topk; ++j) {
      const int32_t i = idx[n * (int64_t)topk + j];
      if (i == -1) continue;
      if (i < 0 || i >= kv_len || (int64_t)(i / page_size) >= num_logical_pages) {
        bad += 1;
        continue;
      }
      const int32_t pg = page_table[i / page_size];
      if (pg < 0 || pg >= num_pages) {
        bad += 1;
        continue;
      }
      list[cnt++] = i;
    }
    qsort(list, (size_t)cnt, sizeof(int32_t), cmp_i32);
    for (int h = 0; h < H; ++h) {
      double* o = out + (n * H + h) * (int64_t)dv;
      for (int t = 0; t < dv; ++t) o[t] = 0.0;
      if (cnt == 0) {
        lse[n * H + h] = -INFINITY;
        continue;
      }
      const float* qh = q + (n * H + h) * (int64_t)dqk;
      double m = -INFINITY;
      for (int j = 0; j < cnt; ++j) {
        const int32_t i = list[j];
        const float* row =
            kv_cache + ((int64_t)page_table[i / page_size] * page_size + i % page_size) * dqk;
        double acc = 0.0;
        for (int t = 0; t < dqk; ++t) acc += (double)qh[t] * (double)row[t];
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
      }
      double l = 0.0;
      for (int j = 0; j < cnt; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
      }
      for (int j = 0; j < cnt; ++j) {
        const int32_t i = list[j];
        const float* row =
            kv_cache + ((int64_t)page_table[i / page_size] * page_size + i % page_size) * dqk;
        const double p = s[j] / l;
        for (int t = 0; t < dv; ++t) o[t] += p * (double)row[t];
      }
      lse[n * H + h] = m + log(l);
    }
    free(list);
    free(s);
  }
  return bad;
}

/* ------------------------------------------------------------------------ */
/* O4. Vision-encoder QKV projection + RoPE ("DeepSeek V4.1 上 4×RTX 3090",   */
/* 坑 1: the qkv + RoPE step checked block by block against a CPU reference; */
/* the position-indexed cos/sin cache of "从 SGLang Kernel源码到 GPU Trace",  */
/* section 3.3). The pages leave the RoPE variant open; the reading taken:   */
/* one-dimensional rotary embedding of every q and k head, rotate-half pairs */
/* (j, j + d/2), angle pos * base^(-2j/d).                                   */
/*                                                                           */
/* x    [n, hidden]; w [3 * heads * d, hidden] (rows: q heads, k heads, v    */
/*      heads); bias [3 * heads * d] or NULL; pos [n].                        */
/* q, k, v [n, heads, d] (double). Plain loops: y = w x + bias, then each q  */
/* and k head rotated pair by pair; v as projected.                          */
/* ------------------------------------------------------------------------ */
void oracle_qkv_rope(const float* x, int64_t n, int hidden, const float* w, const float* bias,
                     int heads, int d, const int32_t* pos, double base, double* q, double* k,
                     double* v) {
  const int64_t cols = 3LL * heads * d;
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t t = 0; t < n; ++t) {
    double* y = (double*)malloc(sizeof(double) * (size_t)cols);
    for (int64_t c = 0; c < cols; ++c) {
      double s = bias ? (double)bias[c] : 0.0;
      for (int i = 0; i < hidden; ++i) s += (double)w[c * hidden + i] * (double)x[t * hidden + i];
      y[c] = s;
    }
    for (int part = 0; part < 3; ++part) {
      double* dst = part == 0 ? q : (part == 1 ? k : v);
      for (int h = 0; h < heads; ++h) {
        const double* src = y + ((int64_t)part * heads + h) * d;
        double* o = dst + (t * heads + h) * (int64_t)d;
        if (part == 2) {
          for (int i = 0; i < d; ++i) o[i] = src[i];
          continue;
        }
        for (int j = 0; j < d / 2; ++j) {
          const double ang = (double)pos[t] * pow(base, -2.0 * j / d);
          const double c = cos(ang), s = sin(ang);
          const double a = src[j], b = src[j + d / 2];
          o[j] = a * c - b * s;
          o[j + d / 2] = a * s + b * c;
        }
      }
    }
    free(y);
  }
}

/* The cos/sin cache: out[p, j] = (cos, sin)(p * base^(-2j/rot_dim)), p < max_pos. */
void oracle_rope_cache(int max_pos, int rot_dim, double base, double* out) {
  for (int p = 0; p < max_pos; ++p)
    for (int j = 0; j < rot_dim / 2; ++j) {
      const double ang = (double)p * pow(base, -2.0 * j / rot_dim);
      out[((int64_t)p * (rot_dim / 2) + j) * 2] = cos(ang);
      out[((int64_t)p * (rot_dim / 2) + j) * 2 + 1] = sin(ang);
    }
}

/* ------------------------------------------------------------------------ */
/* O5. FP8 (e4m3) block quantization for the prefill QK^T product            */
/* ("从 SGLang Kernel源码到 GPU Trace", section 3.2: part of the prefill runs  */
/* in FP8; "AMD MI250部署DeepSeek-V4-Flash", section 4.1: matmul inputs may   */
/* be FP8 with FP32 accumulation, section 5.3: FP8 by block quantization).    */
/* The pages fix neither the format nor the blocks; the reading taken: e4m3  */
/* (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities, */
/* largest finite value 1.75 * 2^8 = 448, smallest normal 2^-6, subnormals   */
/* j * 2^-9), one fp32 scale per block = (block's max |x|) / 448 in fp32.     */
/* ------------------------------------------------------------------------ */

/* Nearest e4m3 value of x, ties to the even mantissa, magnitudes beyond 448  */
/* clamped to 448. The grid spacing in the binade [2^e, 2^(e+1)) is          */
/* 2^(e-3) for e >= -6, and 2^-9 below 2^-6 (subnormals).                    */
double oracle_round_e4m3(double x) {
  const double a = fabs(x);
  if (a == 0.0) return x;
  int e;
  frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): binade [2^(e-1), 2^e) */
  int eb = e - 1;
  if (eb < -6) eb = -6;
  const double ulp = ldexp(1.0, eb - 3);
  double r = nearbyint(a / ulp) * ulp; /* default rounding mode: to nearest, ties to even */
  if (r > 448.0) r = 448.0;
  return x < 0 ? -r : r;
}

/* Quantize nblocks contiguous blocks of len values: scale[b] = max|x| / 448   */
/* (fp32; 1 for an all-zero block), code = e4m3(x / scale[b]) with the        */
/* division in fp32 (the precision in which the CUDA path takes the same      */
/* decision). codes receives the e4m3 values as floats (exactly).             */
void oracle_quant_e4m3(const float* x, int64_t nblocks, int64_t len, float* scale, float* codes) {
  for (int64_t b = 0; b < nblocks; ++b) {
    const float* xb = x + b * len;
    float amax = 0.f;
    for (int64_t i = 0; i < len; ++i) {
      const float v = fabsf(xb[i]);
      if (v > amax) amax = v;
    }
    const float s = amax > 0.f ? amax / 448.0f : 1.0f;
    scale[b] = s;
    for (int64_t i = 0; i < len; ++i) {
      const float y = xb[i] / s;
      codes[b * len + i] = (float)oracle_round_e4m3((double)y);
    }
  }
}
