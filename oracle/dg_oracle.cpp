// Test infrastructure, not product code.
//
// A plain CPU restatement of one uniform-state denoising step of a
// DiffusionGemma-style block-diffusion decoder, of the annealed denoising loop
// around it and of the block commit.  Only the test-suite, the smoke check and
// the CPU-baseline leg of the benchmark load this file; the device library
// shares no code, header, table or helper with it.
//
// Everything is computed in double precision with straight loops and no
// blocking, fusion or online rescaling.  Where the device path stores a GEMM
// operand in bf16, this file rounds the same quantity to bf16 (round to nearest
// even) when `mirror_bf16` is set, so that both sides see the same operands.
// The optional `nthreads` argument only splits independent outer loops (rows,
// heads) between threads; every per-row result is computed in the same order
// whatever the thread count, so outputs are bit-identical for any `nthreads`.
//
// Sources (page title, then section):
//   [TR]  "DiffusionGemma Technical Report" summary page, section "Method step
//         details" (inference steps 1-5) and its reproduction paragraph that
//         lists the sampler hyper-parameters (Table 2 of the report).
//   [EXP] "DiffusionGemma explained" (Gemma docs), sections "Uniform State
//         Diffusion", "Self-conditioning" and "Architecture: incremental
//         prefill and denoising".
//   [CH12] "DiffusionGemma" chapter of the diffusion docs (12_diffusion_gemma),
//         the KV-cache timing and attention-mask lists and the data-flow
//         pseudocode.
//   [PHX] Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
//         1, 2, 3", SC'11 (Philox4x64-10).
//   The one-layer synthetic stand-in (RMSNorm of embedding + self-conditioning,
//   GQA attention with RoPE, tied LM head with per-position sharpness alpha,
//   FFW of p0.E, Philox keyed by (seed, step, position)) follows the problem
//   statement of this project; the readings of what the pages leave open are
//   written next to each function.
//
// Parity status: every function below is pinned by a CPU test (see the tests
// named in each comment); none is "parity unpinned".

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------- threading --
template <class F>
void parallel_rows(int64_t n, int nthreads, F fn) {
  if (nthreads <= 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  int64_t nt = std::min<int64_t>(nthreads, n);
  std::vector<std::thread> pool;
  for (int64_t t = 0; t < nt; ++t) {
    pool.emplace_back([=]() {
      for (int64_t i = t; i < n; i += nt) fn(i);
    });
  }
  for (auto& th : pool) th.join();
}

// ------------------------------------------------------------ bf16 rounding --
// Round a double to the nearest bfloat16 value (8 significant bits, the float32
// exponent range), ties to even.  Done directly from the double so there is no
// intermediate float rounding.
double round_bf16(double x) {
  if (x == 0.0 || !std::isfinite(x)) return x;
  int e;
  double f = std::frexp(x, &e);  // x = f * 2^e, 0.5 <= |f| < 1
  // bf16 normals have exponents e-1 >= -126; below that the spacing is 2^-133.
  int bits = 8;
  if (e - 1 < -126) bits = 8 - (-126 - (e - 1));
  if (bits < 0) return std::copysign(0.0, x);
  double scaled = std::ldexp(f, bits);
  double r = std::nearbyint(scaled);  // default rounding mode: ties to even
  double y = std::ldexp(r, e - bits);
  if (std::fabs(y) > 3.3895313892515355e38) y = std::copysign(INFINITY, x);
  return y;
}

inline double maybe_bf16(double x, int mirror) { return mirror ? round_bf16(x) : x; }

// ---------------------------------------------------------------- E4M3 ----
// The 8-bit floating-point format E4M3 of the FP8 LM head: sign, 4 exponent
// bits biased by 7, 3 mantissa bits; no infinities, the all-ones pattern is
// NaN, so the largest finite magnitude is 1.75 * 2^8 = 448; subnormals step by
// 2^-9.  Rounding is to nearest, ties to even, saturating at 448 (values that
// would round past it become 448).
double round_e4m3(double x) {
  if (x == 0.0 || std::isnan(x)) return x;
  const double a = std::fabs(x);
  double r;
  if (a >= 464.0) {
    r = 448.0;  // 464 is the midpoint between 448 and the first value past the range
  } else {
    int e;
    std::frexp(a, &e);  // a = f 2^e, 0.5 <= f < 1: the leading bit is 2^(e-1)
    const int lead = e - 1 < -6 ? -6 : e - 1;  // subnormals share the exponent of 2^-6
    const double q = std::ldexp(1.0, lead - 3);
    r = std::nearbyint(a / q) * q;  // a / q is exact (a power-of-two scale)
    if (r > 448.0) r = 448.0;
  }
  return std::copysign(r, x);
}

// The bit pattern of an E4M3 value produced by round_e4m3 (the sign of a zero
// result is kept).
uint8_t e4m3_bits(double r, bool negative) {
  const uint8_t sign = negative ? 0x80 : 0x00;
  const double a = std::fabs(r);
  if (a == 0.0) return sign;
  int e;
  std::frexp(a, &e);
  const int E = e - 1;
  if (E < -6) return sign | (uint8_t)std::lrint(a / std::ldexp(1.0, -9));  // subnormal: m 2^-9
  const int m = (int)std::lrint((a / std::ldexp(1.0, E) - 1.0) * 8.0);
  return sign | (uint8_t)((E + 7) << 3) | (uint8_t)m;
}

double e4m3_value(uint8_t b) {
  const int sign = b >> 7, E = (b >> 3) & 15, m = b & 7;
  const double a = E == 0 ? std::ldexp((double)m, -9) : std::ldexp(1.0 + m / 8.0, E - 7);
  return sign ? -a : a;
}

}  // namespace

extern "C" void or_quantize_rows_e4m3(const float* X, int64_t R, int64_t d, uint8_t* Q, float* scale);

extern "C" {

// ------------------------------------------------------------------ Philox --
// Philox4x64 with 10 rounds [PHX]: each round multiplies counter words 0 and 2
// by the two Philox multipliers, mixes the high halves with words 1 and 3 and
// the round key, and the key is bumped by the two Weyl constants between
// rounds.  Pinned by test_oracle_pins.py::test_philox_matches_numpy and the
// published known answer in tests/golden/philox4x64_10_kat.txt.
void or_philox4x64_10(const uint64_t ctr_in[4], const uint64_t key_in[2], uint64_t out[4]) {
  const uint64_t M0 = 0xD2E7470EE14C6C93ULL, M1 = 0xCA5A826395121157ULL;
  const uint64_t W0 = 0x9E3779B97F4A7C15ULL, W1 = 0xBB67AE8584CAA73BULL;
  uint64_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint64_t k0 = key_in[0], k1 = key_in[1];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) { k0 += W0; k1 += W1; }
    unsigned __int128 p0 = (unsigned __int128)M0 * c0;
    unsigned __int128 p1 = (unsigned __int128)M1 * c2;
    uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
    uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
    uint64_t n0 = hi1 ^ c1 ^ k0;
    uint64_t n1 = lo1;
    uint64_t n2 = hi0 ^ c3 ^ k1;
    uint64_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

// The counter layout that keys every random draw of the method by
// (seed, block, step, canvas, position, vocabulary index, stream):
//   key     = (seed, 0)
//   counter = (v >> 2, pos, (block << 32) | step, (batch << 32) | stream)
//   word    = v & 3
// stream 0 = Gumbel noise of accepted positions, 1 = renoise token,
// 2 = initial canvas.  The pages only say "Philox keyed by (seed, step, pos)";
// this layout is this project's reading, shared by both sides as a definition.
uint64_t or_philox_word(uint64_t seed, int32_t block, int32_t step, int32_t batch, int32_t pos,
                        int64_t v, int32_t stream) {
  uint64_t ctr[4] = {(uint64_t)v >> 2, (uint64_t)(uint32_t)pos,
                     ((uint64_t)(uint32_t)block << 32) | (uint32_t)step,
                     ((uint64_t)(uint32_t)batch << 32) | (uint32_t)stream};
  uint64_t key[2] = {seed, 0};
  uint64_t out[4];
  or_philox4x64_10(ctr, key, out);
  return out[v & 3];
}

// A token drawn uniformly from [0, V): floor(w * V / 2^64), the high word of
// the 128-bit product (exact; no modulo bias beyond 2^-64 V).
int32_t or_uniform_token(uint64_t w, int32_t V) {
  unsigned __int128 p = (unsigned __int128)w * (uint64_t)V;
  return (int32_t)(uint64_t)(p >> 64);
}

// Standard Gumbel noise from one 64-bit word: U = (top 23 bits + 1/2) / 2^23,
// exactly representable in float and strictly inside (0, 1), so G is finite
// (-2.81 <= G <= 16.64); G = -log(-log U).  Evaluated in float, the precision
// the device kernel uses to take the same decision.
float or_gumbel(uint64_t w) {
  float u = ((float)(uint32_t)(w >> 41) + 0.5f) * (1.0f / 8388608.0f);
  return -logf(-logf(u));
}

// Gumbel-max sample of a row of tempered logits s (length V): the index that
// maximises s_v + G_v with G_v the Gumbel noise of word (seed, block, step,
// batch, pos, v, stream 0); ties to the lowest index.  *gap receives the
// difference between the two largest perturbed scores.  Pinned by
// test_gumbel_max_law (chi-square against softmax(s)).
int32_t or_gumbel_argmax(const double* s, int64_t V, uint64_t seed, int32_t block, int32_t step,
                         int32_t batch, int32_t pos, double* gap) {
  double best = -INFINITY, second = -INFINITY;
  int64_t bi = 0;
  for (int64_t v = 0; v < V; ++v) {
    double sc = s[v] + (double)or_gumbel(or_philox_word(seed, block, step, batch, pos, v, 0));
    if (sc > best) { second = best; best = sc; bi = v; }
    else if (sc > second) second = sc;
  }
  if (gap) *gap = best - second;
  return (int32_t)bi;
}

// Many Gumbel-max samples of one row, one per position 0..npos-1 (test helper).
void or_gumbel_argmax_many(const double* s, int64_t V, uint64_t seed, int32_t npos, int32_t* out) {
  for (int32_t p = 0; p < npos; ++p) out[p] = or_gumbel_argmax(s, V, seed, 0, 0, 0, p, nullptr);
}

// Many uniform tokens, one per position 0..npos-1 of stream 1 (test helper).
void or_uniform_many(int32_t V, uint64_t seed, int32_t npos, int32_t* out) {
  for (int32_t p = 0; p < npos; ++p) out[p] = or_uniform_token(or_philox_word(seed, 0, 0, 0, p, 0, 1), V);
}

// Many Gumbel values, for words of stream 0 at vocabulary indices 0..n-1 (test helper).
void or_gumbel_many(uint64_t seed, int64_t n, float* out) {
  for (int64_t v = 0; v < n; ++v) out[v] = or_gumbel(or_philox_word(seed, 0, 0, 0, 0, v, 0));
}

// Initial canvas: C tokens drawn uniformly over the vocabulary, [TR] step 2
// ("x_1 sampled uniformly from the vocabulary, z_1 = 0"); stream 2.
void or_canvas_init(int32_t* tokens, int32_t B, int32_t C, int32_t V, uint64_t seed, int32_t block) {
  for (int32_t b = 0; b < B; ++b)
    for (int32_t i = 0; i < C; ++i)
      tokens[(int64_t)b * C + i] = or_uniform_token(or_philox_word(seed, block, 0, b, i, 0, 2), V);
}

// ------------------------------------------------------- small definitions --
// RMS normalisation without a learned gain: y = x / sqrt(mean(x^2) + eps).
// Pinned by test_rmsnorm_unit_rms.
void or_rmsnorm(const double* x, int32_t n, double eps, double* y) {
  double ss = 0.0;
  for (int32_t j = 0; j < n; ++j) ss += x[j] * x[j];
  double r = 1.0 / std::sqrt(ss / n + eps);
  for (int32_t j = 0; j < n; ++j) y[j] = x[j] * r;
}

// Rotary position embedding, half-split pairing: element j is paired with
// j + hd/2 and the pair is rotated by pos * base^(-2j/hd).  Pinned by
// test_rope_* (norm preservation, relative-position property, complex form).
void or_rope(double* x, int32_t hd, double pos, double base) {
  int32_t half = hd / 2;
  for (int32_t j = 0; j < half; ++j) {
    double theta = std::pow(base, -2.0 * j / hd);
    double ang = pos * theta;
    double c = std::cos(ang), s = std::sin(ang);
    double x0 = x[j], x1 = x[j + half];
    x[j] = x0 * c - x1 * s;
    x[j + half] = x0 * s + x1 * c;
  }
}

// GELU with the exact erf form: 0.5 x (1 + erf(x / sqrt 2)).  Pinned against
// torch.nn.functional.gelu in test_gelu_matches_torch.
double or_gelu(double x) { return 0.5 * x * (1.0 + std::erf(x / std::sqrt(2.0))); }

// Tempered softmax statistics of one row of logits l (length V) at
// temperature tau, [TR] step 3: s = l / tau, m = max s, Z = sum exp(s - m),
// S = sum exp(s - m)(s - m), entropy H = log Z - S / Z (nats, = -sum p log p),
// argmax over l with ties to the lowest index, and the gap between the two
// largest logits.  Pinned by test_entropy_* (uniform row gives log V,
// two-level closed form, agreement with scipy.stats.entropy).
void or_row_stats(const double* l, int64_t V, double tau, double* H, double* m_out, double* Z_out,
                  int32_t* argmax, double* top2gap) {
  double m = -INFINITY;
  int64_t am = 0;
  double best = -INFINITY, second = -INFINITY;
  for (int64_t v = 0; v < V; ++v) {
    double s = l[v] / tau;
    if (s > m) m = s;
    if (l[v] > best) { second = best; best = l[v]; am = v; }
    else if (l[v] > second) second = l[v];
  }
  double Z = 0.0, S = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    double t = l[v] / tau - m;
    double e = std::exp(t);
    if (e > 0.0) {  // an excluded entry (l = -inf) has p = 0 and adds nothing
      Z += e;
      S += e * t;
    }
  }
  if (H) *H = std::log(Z) - S / Z;
  if (m_out) *m_out = m;
  if (Z_out) *Z_out = Z;
  if (argmax) *argmax = (int32_t)am;
  if (top2gap) *top2gap = best - second;
}

// Entropy-bounded acceptance, [TR] step 3: positions are sorted by ascending
// entropy (ties by position) and the longest sorted prefix whose cumulative
// entropy stays within the budget b is accepted.  Returns the number accepted;
// fills accept[i], the cumulative entropy cum[i] at position i's rank and
// rank[i].  Pinned by test_accept_bruteforce (all subsets at C <= 12) and the
// invariant tests.
int32_t or_accept(const double* H, int32_t C, double b, uint8_t* accept, double* cum, int32_t* rank) {
  std::vector<int32_t> order(C);
  for (int32_t i = 0; i < C; ++i) order[i] = i;
  std::sort(order.begin(), order.end(), [&](int32_t x, int32_t y) {
    if (H[x] != H[y]) return H[x] < H[y];
    return x < y;
  });
  double c = 0.0;
  int32_t n = 0;
  bool open = true;
  for (int32_t k = 0; k < C; ++k) {
    int32_t i = order[k];
    c += H[i];
    if (cum) cum[i] = c;
    if (rank) rank[i] = k;
    bool acc = open && c <= b;
    if (!acc) open = false;
    accept[i] = acc ? 1 : 0;
    n += acc ? 1 : 0;
  }
  return n;
}

// Bidirectional attention of one query row against keys/values
// [prefix rows 0..P-1 ; canvas rows 0..C-1] with no mask ([CH12] "current
// canvas: full matrix / bidirectional attention; canvas reads the prompt and
// finished-block KV cache"; [EXP] denoise mode).  Scale 1/sqrt(hd).  Pinned
// against torch scaled_dot_product_attention in test_attention_matches_sdpa.
void or_attend_row(const double* q, const float* Kp, const float* Vp, int64_t P,
                   const double* Kc, const double* Vc, int64_t C, int32_t hd, double* o) {
  std::vector<double> sc(P + C);
  double scale = 1.0 / std::sqrt((double)hd);
  double mx = -INFINITY;
  for (int64_t j = 0; j < P + C; ++j) {
    double acc = 0.0;
    if (j < P) {
      for (int32_t t = 0; t < hd; ++t) acc += q[t] * (double)Kp[j * hd + t];
    } else {
      for (int32_t t = 0; t < hd; ++t) acc += q[t] * Kc[(j - P) * hd + t];
    }
    sc[j] = acc * scale;
    mx = std::max(mx, sc[j]);
  }
  double den = 0.0;
  for (int64_t j = 0; j < P + C; ++j) { sc[j] = std::exp(sc[j] - mx); den += sc[j]; }
  for (int32_t t = 0; t < hd; ++t) o[t] = 0.0;
  for (int64_t j = 0; j < P + C; ++j) {
    double p = sc[j] / den;
    if (j < P) {
      for (int32_t t = 0; t < hd; ++t) o[t] += p * (double)Vp[j * hd + t];
    } else {
      for (int32_t t = 0; t < hd; ++t) o[t] += p * Vc[(j - P) * hd + t];
    }
  }
}

// ------------------------------------------------------------- the step -----
typedef struct {
  int32_t V, d, C, B, Hq, Hkv, hd, F;
  int32_t P;    // prefix length held in the cache (same for every canvas)
  int32_t cap;  // cache row capacity per (canvas, kv head)
  double rope_base, rms_eps;
  int32_t mirror_bf16;
  int32_t L;    // attention layers (>= 1); weights Wq, Wk, Wv, Wo and the caches are stacked [L][...]
  // Mixture-of-experts FFN after each attention block (n_exp = 0: none):
  // n_exp routed experts of hidden width Fe, top_k of them per token, plus one
  // shared expert of the same shape.
  int32_t n_exp, top_k, Fe;
} or_dims;

// Weights of the MoE FFN, stacked per layer: router Wr [L][n_exp][d]; expert
// matrices We1 [L][n_exp + 1][Fe][d] and We2 [L][n_exp + 1][d][Fe], expert
// index n_exp being the shared expert.
typedef struct {
  const float *Wr, *We1, *We2;
} or_moe_w;

typedef struct {
  const float *E, *Wq, *Wk, *Wv, *Wo, *W1, *W2;  // [V][d], [L][out][in] row-major (W1, W2 single)
  const float *Kc, *Vc;                          // prefix caches [L][B][Hkv][cap][hd], keys post-RoPE
  const int32_t* x;                              // canvas tokens x_t [B][C]
  const float* z;                                // self-conditioning z_t [B][C][d]
  const float* alpha;                            // per-position logit sharpness [B][C]
  const int32_t* prev_argmax;                    // argmax of the previous step [B][C], or NULL
  double tau, b, stop_H;
  uint64_t seed;
  int32_t step, block;
  // token excluded from the softmax (its logit taken as -inf), or -1: the
  // [MASK] token of masked confidence decoding, which is not a prediction
  // target
  int32_t exclude_tok;
  // FP8 LM head, or NULL: E8 [V][d] E4M3 codes of E with per-row scales
  // E8_scale [V] (or_quantize_rows_e4m3 of E).  The logits then read h
  // quantized the same way per row: l_v = alpha s_h s_v (q_h . q_v) / sqrt(d).
  // The embedding and the contraction p0 . E keep the bf16 E.
  const uint8_t* E8;
  const float* E8_scale;
  or_moe_w moe;  // used when n_exp > 0
} or_step_in;

typedef struct {
  // Every pointer may be NULL (not wanted).  Row-indexed arrays are [B*C].
  double *a, *q, *k, *v, *o, *h;       // [B*C][d], [B*C][Hq*hd], [B*C][Hkv*hd] x2, [B*C][Hq*hd], [B*C][d]
  double* logits;                      // [B*C][V] in full mode, [nrows][V] (rows order) in rows mode
  double *H, *m, *Z, *top2gap;         // per row
  int32_t* argmax;                     // per row
  uint8_t* accept;                     // per row (full mode)
  double* cum;                         // per row (full mode)
  int32_t* rank;                       // per row (full mode)
  int32_t* renoise_tok;                // per row: the uniform token for the row
  int32_t* sample_tok;                 // per row: the Gumbel-max sample for the row
  double* gumbel_gap;                  // per row: top-two gap of s + G
  int32_t* tokens_out;                 // x_{t+1} [B*C] (full mode)
  double *u, *g, *z_out;               // [B*C][d], [B*C][F], [B*C][d]
  int32_t* n_acc;                      // [B]
  double* meanH;                       // [B]
  int32_t* stop;                       // [B]
  // MoE routing of the last layer (n_exp > 0): expert ids in rank order and
  // their gates, [B*C][top_k]; the router logits [B*C][n_exp]
  int32_t* moe_idx;
  double *moe_gate, *moe_logits;
  double* moe_x;  // the last layer's router input RMSNorm(h) [B*C][d]
} or_step_out;

// ------------------------------------------------------------------ MoE -----
// The mixture-of-experts FFN of one layer, applied to rows h [n][d] in place
// (the DiffusionGemma backbone's FFN: the "文本 Diffusion 模型" survey page,
// §11 -- 128 experts per layer, 8 routed plus one shared -- and §13 -- router
// top-k, expert GEMM, token permutation; the technical report summary's MoE
// paragraph -- each token activates a few experts).  Per row, as a pre-norm residual block:
//   x   = RMSNorm(h)                          (bf16 when mirroring)
//   r_e = x . Wr_e                            router logit of routed expert e
//   S   = the top_k experts by r (ties: lower index first), in rank order
//   g_j = exp(r_{S_j}) / sum_{e in S} exp(r_e)     softmax over the selected
//         logits, i.e. the softmax over all experts renormalised on S
//   y   = sum_j g_j FFN_{S_j}(x) + FFN_shared(x),  FFN_e(x) = We2_e GELU(We1_e x)
//         (no biases; the hidden GELU output rounded to bf16 when mirroring)
//   h  <- h + y                               (bf16 when mirroring)
// The pages give neither the expert width nor the gating formula; the
// softmax-then-top-k-renormalised gate and the two-matrix GELU expert (the
// self-conditioning FFW's shape) are the plainest readings.  Optional outputs:
// idx [n][top_k], gate [n][top_k], logits [n][n_exp], x [n][d] (the router's input).
void moe_ffn(const or_dims* D, const float* Wr, const float* We1, const float* We2, double* h, int64_t n,
             int32_t* idx_out, double* gate_out, double* logit_out, double* x_out, int nthreads) {
  const int64_t d = D->d, NE = D->n_exp, K = D->top_k, Fe = D->Fe;
  const int mir = D->mirror_bf16;
  parallel_rows(n, nthreads, [&](int64_t r) {
    double* hr = &h[r * d];
    std::vector<double> x(d), rl(NE), hid(Fe), y(d, 0.0);
    or_rmsnorm(hr, (int32_t)d, D->rms_eps, x.data());
    for (int64_t j = 0; j < d; ++j) x[j] = maybe_bf16(x[j], mir);
    if (x_out)
      for (int64_t j = 0; j < d; ++j) x_out[r * d + j] = x[j];
    for (int64_t e = 0; e < NE; ++e) {
      double acc = 0.0;
      for (int64_t j = 0; j < d; ++j) acc += x[j] * (double)Wr[e * d + j];
      rl[e] = acc;
    }
    std::vector<int32_t> order(NE);
    for (int64_t e = 0; e < NE; ++e) order[e] = (int32_t)e;
    std::stable_sort(order.begin(), order.end(), [&](int32_t u, int32_t v) { return rl[u] > rl[v]; });
    const double top = rl[order[0]];
    double Z = 0.0;
    for (int64_t j = 0; j < K; ++j) Z += std::exp(rl[order[j]] - top);
    auto expert = [&](int64_t e, double gate) {
      const float* W1 = We1 + e * Fe * d;
      const float* W2 = We2 + e * d * Fe;
      for (int64_t f = 0; f < Fe; ++f) {
        double acc = 0.0;
        for (int64_t j = 0; j < d; ++j) acc += x[j] * (double)W1[f * d + j];
        hid[f] = maybe_bf16(or_gelu(acc), mir);
      }
      for (int64_t c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int64_t f = 0; f < Fe; ++f) acc += hid[f] * (double)W2[c * Fe + f];
        y[c] += gate * acc;
      }
    };
    for (int64_t j = 0; j < K; ++j) {
      const double g = std::exp(rl[order[j]] - top) / Z;
      if (idx_out) idx_out[r * K + j] = order[j];
      if (gate_out) gate_out[r * K + j] = g;
      expert(order[j], g);
    }
    expert(NE, 1.0);  // the shared expert
    if (logit_out)
      for (int64_t e = 0; e < NE; ++e) logit_out[r * NE + e] = rl[e];
    for (int64_t c = 0; c < d; ++c) hr[c] = maybe_bf16(hr[c] + y[c], mir);
  });
}

// One denoising step, [TR] step 3 (and the stop test of step 4):
//   a1  a = RMSNorm(E[x_t] + z_t)                       [CH12] pseudocode, [TR]
//   a2  q = RoPE(a Wq^T), k = RoPE(a Wk^T), v = a Wv^T  (positions P + i)
//   a3  o = softmax(q [K_pre; k]^T / sqrt(hd)) [V_pre; v], no mask, GQA
//   a4  h = a + o Wo^T
//   a5  l = alpha_i (h E^T) / sqrt(d); p0 = softmax(l / tau); entropy; argmax
//   a6  accept the entropy-sorted prefix within budget b; renoise the rest
//   a7  accepted positions take the Gumbel-max sample of s = l / tau
//   a8  u = p0 E                                          [EXP] self-conditioning
//   a9  z_{t+1} = W2 GELU(W1 u)                           [TR] z = FFW(p0 E)
//   a10 stop when mean entropy <= stop_H and argmax equals the previous step's
//
// `rows`/`nrows`: when rows != NULL only those global rows (b*C + i) get a5,
// a7, a8 and a9 (for large vocabularies), and the acceptance a6 is skipped.
// Returns 0 on success, 1 on bad arguments.
int or_denoise_step(const or_dims* D, const or_step_in* in, or_step_out* out, const int32_t* rows,
                    int32_t nrows, int32_t nthreads) {
  if (!D || !in || !out) return 1;
  const int64_t V = D->V, d = D->d, C = D->C, B = D->B, Hq = D->Hq, Hkv = D->Hkv, hd = D->hd,
                F = D->F, P = D->P, cap = D->cap;
  if (V <= 0 || d <= 0 || C <= 0 || B <= 0 || Hq <= 0 || Hkv <= 0 || hd <= 0 || F <= 0 ||
      Hq % Hkv != 0 || hd % 2 != 0 || P < 0 || P > cap)
    return 1;
  if (D->n_exp < 0 || (D->n_exp > 0 && (D->top_k < 1 || D->top_k > D->n_exp || D->Fe < 1 || !in->moe.Wr ||
                                        !in->moe.We1 || !in->moe.We2)))
    return 1;
  const int mir = D->mirror_bf16;
  const int64_t M = B * C, nq = Hq * hd, nkv = Hkv * hd;

  // a1: embedding of the current canvas plus the self-conditioning vector,
  // then RMSNorm.
  std::vector<double> a(M * d);
  parallel_rows(M, nthreads, [&](int64_t r) {
    std::vector<double> e(d);
    int64_t tok = in->x[r];
    for (int64_t j = 0; j < d; ++j) e[j] = (double)in->E[tok * d + j] + (double)in->z[r * d + j];
    or_rmsnorm(e.data(), (int32_t)d, D->rms_eps, &a[r * d]);
    for (int64_t j = 0; j < d; ++j) a[r * d + j] = maybe_bf16(a[r * d + j], mir);
  });

  // a2-a4, once per attention layer.  The one-layer stand-in generalises as
  // pre-norm residual blocks (a reading: the pages' model has 30 layers, the
  // stand-in's layer is fixed by the problem statement): layer l takes a_l,
  // h_l = a_l + Attn_l(a_l) Wo_l^T, and a_{l+1} = RMSNorm(h_l); the LM head
  // reads h_{L-1}.  Layer l attends over its own prefix cache.  With L = 1
  // this is exactly the single layer.  The debug copies are the last layer's.
  const int64_t L = D->L < 1 ? 1 : D->L;
  std::vector<double> q(M * nq), k(M * nkv), v(M * nkv), o(M * nq), hh(M * d);
  for (int64_t l = 0; l < L; ++l) {
    const float* Wq = in->Wq + l * nq * d;
    const float* Wk = in->Wk + l * nkv * d;
    const float* Wv = in->Wv + l * nkv * d;
    const float* Wo = in->Wo + l * d * nq;
    const float* Kcl = in->Kc + l * B * Hkv * cap * hd;
    const float* Vcl = in->Vc + l * B * Hkv * cap * hd;
    if (l > 0) {
      parallel_rows(M, nthreads, [&](int64_t r) {
        or_rmsnorm(&hh[r * d], (int32_t)d, D->rms_eps, &a[r * d]);
        for (int64_t j = 0; j < d; ++j) a[r * d + j] = maybe_bf16(a[r * d + j], mir);
      });
    }
    // a2: projections; RoPE on q and k at absolute position P + i.
    parallel_rows(M, nthreads, [&](int64_t r) {
      const double* ar = &a[r * d];
      double pos = (double)(P + r % C);
      for (int64_t n = 0; n < nq; ++n) {
        double acc = 0.0;
        for (int64_t j = 0; j < d; ++j) acc += ar[j] * (double)Wq[n * d + j];
        q[r * nq + n] = acc;
      }
      for (int64_t n = 0; n < nkv; ++n) {
        double acc = 0.0, acc2 = 0.0;
        for (int64_t j = 0; j < d; ++j) {
          acc += ar[j] * (double)Wk[n * d + j];
          acc2 += ar[j] * (double)Wv[n * d + j];
        }
        k[r * nkv + n] = acc;
        v[r * nkv + n] = acc2;
      }
      for (int64_t h = 0; h < Hq; ++h) or_rope(&q[r * nq + h * hd], (int32_t)hd, pos, D->rope_base);
      for (int64_t h = 0; h < Hkv; ++h) or_rope(&k[r * nkv + h * hd], (int32_t)hd, pos, D->rope_base);
      for (int64_t n = 0; n < nq; ++n) q[r * nq + n] = maybe_bf16(q[r * nq + n], mir);
      for (int64_t n = 0; n < nkv; ++n) {
        k[r * nkv + n] = maybe_bf16(k[r * nkv + n], mir);
        v[r * nkv + n] = maybe_bf16(v[r * nkv + n], mir);
      }
    });

    // a3: bidirectional GQA attention over [prefix cache ; canvas].  Query head
    // h reads kv head h / (Hq / Hkv).
    parallel_rows(B * Hq, nthreads, [&](int64_t bh) {
      int64_t bb = bh / Hq, h = bh % Hq, g = h / (Hq / Hkv);
      std::vector<double> kc(C * hd), vc(C * hd), qr(hd), orow(hd);
      for (int64_t i = 0; i < C; ++i)
        for (int64_t t = 0; t < hd; ++t) {
          kc[i * hd + t] = k[(bb * C + i) * nkv + g * hd + t];
          vc[i * hd + t] = v[(bb * C + i) * nkv + g * hd + t];
        }
      const float* Kp = Kcl + ((bb * Hkv + g) * cap) * hd;
      const float* Vp = Vcl + ((bb * Hkv + g) * cap) * hd;
      for (int64_t i = 0; i < C; ++i) {
        for (int64_t t = 0; t < hd; ++t) qr[t] = q[(bb * C + i) * nq + h * hd + t];
        or_attend_row(qr.data(), Kp, Vp, P, kc.data(), vc.data(), C, (int32_t)hd, orow.data());
        for (int64_t t = 0; t < hd; ++t) o[(bb * C + i) * nq + h * hd + t] = maybe_bf16(orow[t], mir);
      }
    });

    // a4: output projection with the residual from a.
    parallel_rows(M, nthreads, [&](int64_t r) {
      for (int64_t n = 0; n < d; ++n) {
        double acc = 0.0;
        for (int64_t j = 0; j < nq; ++j) acc += o[r * nq + j] * (double)Wo[n * nq + j];
        hh[r * d + n] = maybe_bf16(a[r * d + n] + acc, mir);
      }
    });
    // the layer's MoE FFN (when configured); the routing outputs are the last layer's
    if (D->n_exp > 0) {
      const bool lastl = l == L - 1;
      moe_ffn(D, in->moe.Wr + l * D->n_exp * d, in->moe.We1 + l * (D->n_exp + 1) * (int64_t)D->Fe * d,
              in->moe.We2 + l * (D->n_exp + 1) * d * (int64_t)D->Fe, hh.data(), M,
              lastl ? out->moe_idx : nullptr, lastl ? out->moe_gate : nullptr,
              lastl ? out->moe_logits : nullptr, lastl ? out->moe_x : nullptr, nthreads);
    }
  }

  if (out->a) std::memcpy(out->a, a.data(), sizeof(double) * M * d);
  if (out->q) std::memcpy(out->q, q.data(), sizeof(double) * M * nq);
  if (out->k) std::memcpy(out->k, k.data(), sizeof(double) * M * nkv);
  if (out->v) std::memcpy(out->v, v.data(), sizeof(double) * M * nkv);
  if (out->o) std::memcpy(out->o, o.data(), sizeof(double) * M * nq);
  if (out->h) std::memcpy(out->h, hh.data(), sizeof(double) * M * d);

  // Rows that get the vocabulary stages.
  std::vector<int64_t> rl;
  if (rows) {
    for (int32_t t = 0; t < nrows; ++t) {
      if (rows[t] < 0 || rows[t] >= M) return 1;
      rl.push_back(rows[t]);
    }
  } else {
    for (int64_t r = 0; r < M; ++r) rl.push_back(r);
  }
  const bool full = (rows == nullptr);
  const double inv_sqrt_d = 1.0 / std::sqrt((double)d);

  // a5 + a7 + a8 per row.  The logits row is rebuilt here from its definition.
  std::vector<double> Hrow(M, 0.0), mrow(M, 0.0), Zrow(M, 0.0), gap(M, 0.0), ggap(M, 0.0);
  std::vector<int32_t> am(M, 0), samp(M, 0);
  std::vector<double> u(M * d, 0.0);
  parallel_rows((int64_t)rl.size(), nthreads, [&](int64_t t) {
    int64_t r = rl[t];
    int64_t bb = r / C, i = r % C;
    std::vector<double> lrow(V);
    const double* hr = &hh[r * d];
    double al = (double)in->alpha[r];
    if (in->E8) {
      // FP8 head: h quantized per row (h is bf16-representable, so float exact)
      std::vector<float> hf(d);
      std::vector<uint8_t> hq(d);
      float hs;
      for (int64_t j = 0; j < d; ++j) hf[j] = (float)hr[j];
      or_quantize_rows_e4m3(hf.data(), 1, d, hq.data(), &hs);
      std::vector<double> hv(d);
      for (int64_t j = 0; j < d; ++j) hv[j] = e4m3_value(hq[j]);
      for (int64_t vv = 0; vv < V; ++vv) {
        double acc = 0.0;
        for (int64_t j = 0; j < d; ++j) acc += hv[j] * e4m3_value(in->E8[vv * d + j]);
        lrow[vv] = al * ((double)hs * (double)in->E8_scale[vv] * acc) * inv_sqrt_d;
      }
    } else {
      for (int64_t vv = 0; vv < V; ++vv) {
        double acc = 0.0;
        for (int64_t j = 0; j < d; ++j) acc += hr[j] * (double)in->E[vv * d + j];
        lrow[vv] = al * acc * inv_sqrt_d;
      }
    }
    if (out->logits) std::memcpy(&out->logits[(full ? r : t) * V], lrow.data(), sizeof(double) * V);
    if (in->exclude_tok >= 0 && in->exclude_tok < V) lrow[in->exclude_tok] = -INFINITY;
    double Hv, mv, Zv, g2;
    int32_t a_m;
    or_row_stats(lrow.data(), V, in->tau, &Hv, &mv, &Zv, &a_m, &g2);
    Hrow[r] = Hv; mrow[r] = mv; Zrow[r] = Zv; am[r] = a_m; gap[r] = g2;
    // a7: Gumbel-max sample of s = l / tau (stream 0, vocabulary index v).
    for (int64_t vv = 0; vv < V; ++vv) lrow[vv] /= in->tau;
    double gg;
    samp[r] = or_gumbel_argmax(lrow.data(), V, in->seed, in->block, in->step, (int32_t)bb,
                               (int32_t)i, &gg);
    ggap[r] = gg;
    for (int64_t vv = 0; vv < V; ++vv) lrow[vv] *= in->tau;
    // a8: u = sum_v p0_v E_v with p0 = exp(s - m) / Z.
    double* ur = &u[r * d];
    for (int64_t vv = 0; vv < V; ++vv) {
      double p = std::exp(lrow[vv] / in->tau - mv) / Zv;
      if (p == 0.0) continue;
      for (int64_t j = 0; j < d; ++j) ur[j] += p * (double)in->E[vv * d + j];
    }
    for (int64_t j = 0; j < d; ++j) ur[j] = maybe_bf16(ur[j], mir);
  });

  // a9: z_{t+1} = W2 GELU(W1 u), no biases.
  std::vector<double> g(M * F, 0.0), zo(M * d, 0.0);
  parallel_rows((int64_t)rl.size(), nthreads, [&](int64_t t) {
    int64_t r = rl[t];
    for (int64_t f = 0; f < F; ++f) {
      double acc = 0.0;
      for (int64_t j = 0; j < d; ++j) acc += u[r * d + j] * (double)in->W1[f * d + j];
      g[r * F + f] = maybe_bf16(or_gelu(acc), mir);
    }
    for (int64_t n = 0; n < d; ++n) {
      double acc = 0.0;
      for (int64_t f = 0; f < F; ++f) acc += g[r * F + f] * (double)in->W2[n * F + f];
      zo[r * d + n] = maybe_bf16(acc, mir);
    }
  });

  for (int64_t r : rl) {
    int64_t bb = r / C, i = r % C;
    if (out->H) out->H[r] = Hrow[r];
    if (out->m) out->m[r] = mrow[r];
    if (out->Z) out->Z[r] = Zrow[r];
    if (out->top2gap) out->top2gap[r] = gap[r];
    if (out->argmax) out->argmax[r] = am[r];
    if (out->sample_tok) out->sample_tok[r] = samp[r];
    if (out->gumbel_gap) out->gumbel_gap[r] = ggap[r];
    if (out->renoise_tok)
      out->renoise_tok[r] = or_uniform_token(
          or_philox_word(in->seed, in->block, in->step, (int32_t)bb, (int32_t)i, 0, 1), (int32_t)V);
    if (out->u) std::memcpy(&out->u[r * d], &u[r * d], sizeof(double) * d);
    if (out->g) std::memcpy(&out->g[r * F], &g[r * F], sizeof(double) * F);
    if (out->z_out) std::memcpy(&out->z_out[r * d], &zo[r * d], sizeof(double) * d);
  }
  if (!full) return 0;

  // a6 + a10 per canvas.
  for (int64_t bb = 0; bb < B; ++bb) {
    std::vector<uint8_t> acc(C);
    std::vector<double> cum(C);
    std::vector<int32_t> rk(C);
    int32_t na = or_accept(&Hrow[bb * C], (int32_t)C, in->b, acc.data(), cum.data(), rk.data());
    double sH = 0.0;
    for (int64_t i = 0; i < C; ++i) sH += Hrow[bb * C + i];
    double mH = sH / (double)C;
    bool same = in->prev_argmax != nullptr && in->step >= 1;
    if (same)
      for (int64_t i = 0; i < C; ++i)
        if (in->prev_argmax[bb * C + i] != am[bb * C + i]) { same = false; break; }
    int32_t st = (mH <= in->stop_H && same) ? 1 : 0;
    for (int64_t i = 0; i < C; ++i) {
      int64_t r = bb * C + i;
      if (out->accept) out->accept[r] = acc[i];
      if (out->cum) out->cum[r] = cum[i];
      if (out->rank) out->rank[r] = rk[i];
      if (out->tokens_out)
        out->tokens_out[r] = acc[i] ? samp[r]
                                    : or_uniform_token(or_philox_word(in->seed, in->block, in->step,
                                                                      (int32_t)bb, (int32_t)i, 0, 1),
                                                       (int32_t)V);
    }
    if (out->n_acc) out->n_acc[bb] = na;
    if (out->meanH) out->meanH[bb] = mH;
    if (out->stop) out->stop[bb] = st;
  }
  return 0;
}

// ------------------------------------------- masked confidence decoding ---
// The second sampler, masked confidence decoding ([P4] "从零拆开DiffusionGemma",
// the generate() of its fourth step): the canvas starts as [MASK] everywhere;
// each of N steps predicts every position, takes the confidence of a position
// as the largest tempered probability max_v p0_v = 1 / Z (Z = sum_v
// exp(s_v - max s)) and its candidate as the argmax, and reveals the
// k = min(ceil(U / (N - step)), U) still-masked positions of highest
// confidence (U of them still masked), writing their candidates; revealed
// positions never change again, so after step N - 1 nothing is masked.
// Readings: ties in confidence go to the lower position; the candidate is the
// argmax with the lowest index on ties.
// Z[C], argmax[C], tokens[C] (updated in place), mask_id, step, N.  Fills
// revealed[i] = 1 for the positions revealed by this step.  Returns k, or -1
// on bad arguments.  Pinned by test_oracle_pins.py::test_reveal_matches_topk
// and test_reveal_loop_invariants.
int32_t or_reveal(const double* Z, const int32_t* argmax, int32_t* tokens, int32_t C, int32_t mask_id,
                  int32_t step, int32_t N, uint8_t* revealed) {
  if (C <= 0 || N <= 0 || step < 0 || step >= N) return -1;
  std::vector<int32_t> idx;
  for (int32_t i = 0; i < C; ++i) {
    revealed[i] = 0;
    if (tokens[i] == mask_id) idx.push_back(i);
  }
  const int32_t U = (int32_t)idx.size();
  const int32_t remaining = N - step;
  int32_t k = (U + remaining - 1) / remaining;
  if (k > U) k = U;
  // highest confidence first: smallest Z (confidence 1 / Z), then lower position
  std::stable_sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) { return Z[a] < Z[b]; });
  for (int32_t t = 0; t < k; ++t) {
    tokens[idx[t]] = argmax[idx[t]];
    revealed[idx[t]] = 1;
  }
  return k;
}

// -------------------------------------------------------- the canvas loop ---
// Temperature of step s of the anneal: linear from tau0 at step 0 to tau1 at
// step N - 1 ([TR] Table 2: 0.8 -> 0.4 over N = 48 steps; the endpoint is
// reached at the last step).  Pinned by test_oracle_pins.py::
// test_loop_matches_manual_steps_with_linear_anneal (the loop equals manual
// steps at the printed temperatures).
double or_tau(double tau0, double tau1, int32_t N, int32_t s) {
  return (N > 1) ? tau0 + (tau1 - tau0) * (double)s / (double)(N - 1) : tau0;
}

// Up to N denoising steps with the temperature annealed linearly from tau0 at
// step 0 to tau1 at step N-1 ([TR] step 3 and Table 2: N = 48, 0.8 -> 0.4,
// b = 0.1, stop threshold 0.005); each canvas stops on its own when the stop
// test of [TR] step 4 fires, and is frozen from then on.  The result x0_hat
// of a canvas is the argmax of its last step ([TR] step 5 commits x0_hat).
//
// x, z are updated in place.  steps_taken[B], converged[B], accepted[B][N]
// (accepted count per step, -1 after the canvas stopped), xhat0[B][C].
int or_denoise_canvas(const or_dims* D, const float* E, const float* Wq, const float* Wk,
                      const float* Wv, const float* Wo, const float* W1, const float* W2,
                      const float* Kc, const float* Vc, int32_t* x, float* z, const float* alpha,
                      int32_t N, double tau0, double tau1, double b, double stop_H, uint64_t seed,
                      int32_t block, int32_t* steps_taken, int32_t* converged, int32_t* accepted,
                      int32_t* xhat0, int32_t nthreads) {
  const int64_t B = D->B, C = D->C, d = D->d, M = B * C;
  std::vector<int32_t> prev(M, 0), am(M), tok(M), na(B), st(B);
  std::vector<uint8_t> done(B, 0);
  std::vector<double> zo(M * d);
  for (int64_t bb = 0; bb < B; ++bb) { steps_taken[bb] = 0; converged[bb] = 0; }
  for (int64_t t = 0; t < B * N; ++t) accepted[t] = -1;
  for (int32_t s = 0; s < N; ++s) {
    double tau = or_tau(tau0, tau1, N, s);
    or_step_in in{};
    in.E = E; in.Wq = Wq; in.Wk = Wk; in.Wv = Wv; in.Wo = Wo; in.W1 = W1; in.W2 = W2;
    in.Kc = Kc; in.Vc = Vc; in.x = x; in.z = z; in.alpha = alpha;
    in.prev_argmax = prev.data(); in.tau = tau; in.b = b; in.stop_H = stop_H;
    in.seed = seed; in.step = s; in.block = block; in.exclude_tok = -1;
    or_step_out out{};
    out.argmax = am.data(); out.tokens_out = tok.data(); out.z_out = zo.data();
    out.n_acc = na.data(); out.stop = st.data();
    int rc = or_denoise_step(D, &in, &out, nullptr, 0, nthreads);
    if (rc) return rc;
    bool all_done = true;
    for (int64_t bb = 0; bb < B; ++bb) {
      if (done[bb]) continue;
      for (int64_t i = 0; i < C; ++i) {
        int64_t r = bb * C + i;
        x[r] = tok[r];
        prev[r] = am[r];
        xhat0[r] = am[r];
        for (int64_t j = 0; j < d; ++j) z[r * d + j] = (float)zo[r * d + j];
      }
      accepted[bb * N + s] = na[bb];
      steps_taken[bb] = s + 1;
      if (st[bb]) { done[bb] = 1; converged[bb] = 1; }
      if (!done[bb]) all_done = false;
    }
    if (all_done) break;
  }
  return 0;
}

// ------------------------------------------------- prefill and commit ----
// Causal re-encode of n tokens per canvas appended to the caches at rows
// P..P+n-1: the prompt prefill of [TR] step 1 and [EXP] "Architecture:
// incremental prefill and denoising", and the commit of a finalized block of
// [TR] step 5 and [CH12] (the cache comes from re-encoding the finished block,
// not from the denoiser's states).  The encoder is the denoiser's attention
// stack with no self-conditioning (z = 0) and a causal mask: token i attends to
// every cached row and to the block's tokens 0..i.  Per layer l: a_l, k_l and
// v_l (RoPE at positions P + i) are written to cache l first, then (below the
// last layer) q_l attends over cache rows 0..P+i, h_l = a_l + o_l Wo_l^T and
// a_{l+1} = RMSNorm(h_l).  With one layer the appended K/V depend only on each
// token and its position, so the mask has no effect; with two or more, layer
// l + 1's K/V depend on the attention of layer l over earlier tokens.
// Kc, Vc: [L][B][Hkv][cap][hd], updated in place; tokens [B][n].  Returns 1
// if P + n > cap.  Pinned by test_oracle_pins.py::test_prefill_* (a torch
// composition with an explicit causal mask, the independence of earlier K/V
// from later tokens, chunked prefill equal to one piece).
int or_prefill(const or_dims* D, const float* E, const float* Wq, const float* Wk, const float* Wv,
               const float* Wo, const or_moe_w* moe, const int32_t* tokens, int32_t n, float* Kc, float* Vc,
               int32_t nthreads) {
  const int64_t d = D->d, B = D->B, Hq = D->Hq, Hkv = D->Hkv, hd = D->hd, P = D->P, cap = D->cap;
  const int64_t L = D->L < 1 ? 1 : D->L;
  if (n < 0 || P + n > cap) return 1;
  if (D->n_exp > 0 && L > 1 && (!moe || D->top_k < 1 || D->top_k > D->n_exp || D->Fe < 1)) return 1;
  const int mir = D->mirror_bf16;
  const int64_t nq = Hq * hd, nkv = Hkv * hd, Mn = B * (int64_t)n;
  std::vector<double> a(Mn * d), q(Mn * nq), o(Mn * nq), hh(Mn * d);
  parallel_rows(Mn, nthreads, [&](int64_t r) {
    std::vector<double> e(d);
    for (int64_t j = 0; j < d; ++j) e[j] = (double)E[(int64_t)tokens[r] * d + j];
    or_rmsnorm(e.data(), (int32_t)d, D->rms_eps, &a[r * d]);
    for (int64_t j = 0; j < d; ++j) a[r * d + j] = maybe_bf16(a[r * d + j], mir);
  });
  for (int64_t l = 0; l < L; ++l) {
    const float* Wql = Wq + l * nq * d;
    const float* Wkl = Wk + l * nkv * d;
    const float* Wvl = Wv + l * nkv * d;
    const float* Wol = Wo + l * d * nq;
    float* Kl = Kc + l * B * Hkv * cap * hd;
    float* Vl = Vc + l * B * Hkv * cap * hd;
    const bool last = l == L - 1;
    if (l > 0) {
      parallel_rows(Mn, nthreads, [&](int64_t r) {
        or_rmsnorm(&hh[r * d], (int32_t)d, D->rms_eps, &a[r * d]);
        for (int64_t j = 0; j < d; ++j) a[r * d + j] = maybe_bf16(a[r * d + j], mir);
      });
    }
    parallel_rows(Mn, nthreads, [&](int64_t r) {
      const int64_t bb = r / n, i = r % n;
      const double* ar = &a[r * d];
      std::vector<double> k(nkv), v(nkv);
      for (int64_t c = 0; c < nkv; ++c) {
        double acc = 0.0, acc2 = 0.0;
        for (int64_t j = 0; j < d; ++j) {
          acc += ar[j] * (double)Wkl[c * d + j];
          acc2 += ar[j] * (double)Wvl[c * d + j];
        }
        k[c] = acc;
        v[c] = acc2;
      }
      for (int64_t g = 0; g < Hkv; ++g) or_rope(&k[g * hd], (int32_t)hd, (double)(P + i), D->rope_base);
      for (int64_t g = 0; g < Hkv; ++g)
        for (int64_t t = 0; t < hd; ++t) {
          const int64_t dst = ((bb * Hkv + g) * cap + P + i) * hd + t;
          Kl[dst] = (float)maybe_bf16(k[g * hd + t], mir);
          Vl[dst] = (float)maybe_bf16(v[g * hd + t], mir);
        }
      if (!last) {
        for (int64_t c = 0; c < nq; ++c) {
          double acc = 0.0;
          for (int64_t j = 0; j < d; ++j) acc += ar[j] * (double)Wql[c * d + j];
          q[r * nq + c] = acc;
        }
        for (int64_t h = 0; h < Hq; ++h) or_rope(&q[r * nq + h * hd], (int32_t)hd, (double)(P + i), D->rope_base);
        for (int64_t c = 0; c < nq; ++c) q[r * nq + c] = maybe_bf16(q[r * nq + c], mir);
      }
    });
    if (last) break;
    // causal attention: token i over cache rows 0..P+i (the block's own rows
    // were written above)
    parallel_rows(B * Hq, nthreads, [&](int64_t bh) {
      const int64_t bb = bh / Hq, h = bh % Hq, g = h / (Hq / Hkv);
      const float* Kp = Kl + ((bb * Hkv + g) * cap) * hd;
      const float* Vp = Vl + ((bb * Hkv + g) * cap) * hd;
      std::vector<double> orow(hd);
      for (int64_t i = 0; i < n; ++i) {
        const double* qr = &q[(bb * n + i) * nq + h * hd];
        or_attend_row(qr, Kp, Vp, P + i + 1, nullptr, nullptr, 0, (int32_t)hd, orow.data());
        for (int64_t t = 0; t < hd; ++t) o[(bb * n + i) * nq + h * hd + t] = maybe_bf16(orow[t], mir);
      }
    });
    parallel_rows(Mn, nthreads, [&](int64_t r) {
      for (int64_t c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int64_t j = 0; j < nq; ++j) acc += o[r * nq + j] * (double)Wol[c * nq + j];
        hh[r * d + c] = maybe_bf16(a[r * d + c] + acc, mir);
      }
    });
    // the layer's MoE FFN feeds the next layer's input (the last layer's output
    // is not needed for the cache)
    if (D->n_exp > 0)
      moe_ffn(D, moe->Wr + l * D->n_exp * d, moe->We1 + l * (D->n_exp + 1) * (int64_t)D->Fe * d,
              moe->We2 + l * (D->n_exp + 1) * d * (int64_t)D->Fe, hh.data(), Mn, nullptr, nullptr, nullptr,
              nullptr, nthreads);
  }
  return 0;
}

// The commit of a finalized block of C tokens per canvas (or_prefill with
// n = C).  Kept as its own entry for the one-layer callers (Wq, Wo unused
// when L = 1).
int or_commit(const or_dims* D, const float* E, const float* Wk, const float* Wv,
              const int32_t* tokens, float* Kc, float* Vc, int32_t nthreads) {
  if (D->L > 1) return 1;
  return or_prefill(D, E, nullptr, Wk, Wv, nullptr, nullptr, tokens, D->C, Kc, Vc, nthreads);
}

// The MoE FFN of one layer on rows h [n][d] (in place), with its routing.
int or_moe_ffn(const or_dims* D, const float* Wr, const float* We1, const float* We2, double* h, int64_t n,
               int32_t* idx, double* gate, double* logits, int32_t nthreads) {
  if (!D || D->n_exp < 1 || D->top_k < 1 || D->top_k > D->n_exp || D->Fe < 1 || !Wr || !We1 || !We2 || n < 0)
    return 1;
  moe_ffn(D, Wr, We1, We2, h, n, idx, gate, logits, nullptr, nthreads);
  return 0;
}

double or_round_bf16(double x) { return round_bf16(x); }

double or_round_e4m3(double x) { return round_e4m3(x); }
double or_e4m3_value(uint8_t b) { return e4m3_value(b); }

// Per-row quantization to E4M3 with one scale per row (the FP8 LM head's
// operands: its A rows h and its B rows E): scale = absmax / 448 and
// q_j = E4M3(x_j * (448 / absmax)), both quotients and the product rounded to
// float32 (the arithmetic is fixed to float32 so that every implementation of
// this definition gives the same bytes); x_j ~= q_j * scale.  A zero row has
// scale 0 and zero codes.  Pinned by test_quantize_rows_e4m3_matches_torch.
void or_quantize_rows_e4m3(const float* X, int64_t R, int64_t d, uint8_t* Q, float* scale) {
  for (int64_t r = 0; r < R; ++r) {
    const float* x = X + r * d;
    float amax = 0.0f;
    for (int64_t j = 0; j < d; ++j) amax = std::max(amax, std::fabs(x[j]));
    if (!(amax > 0.0f)) {
      scale[r] = 0.0f;
      for (int64_t j = 0; j < d; ++j) Q[r * d + j] = 0;
      continue;
    }
    const float sc = amax / 448.0f;
    const float inv = 448.0f / amax;
    scale[r] = sc;
    for (int64_t j = 0; j < d; ++j) {
      const float xs = x[j] * inv;
      Q[r * d + j] = e4m3_bits(round_e4m3((double)xs), std::signbit(xs));
    }
  }
}

}  // extern "C"
