// Plain fp64 CPU oracle of the MoE-layer forward (sqrt-softplus router or hash router,
// MXFP8 activations, MXFP4 experts, SwiGLU with clamp, weighted combine).
//
// TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's CPU
// baseline leg may load this library.  It shares no code with the CUDA path.
//
// Sources it follows (DeepSeek-V4-Flash pages):
//  * "TensorSharp DeepSeek V4 Flash" page, section "How TensorSharp runs it": the routed
//    experts are chosen by "sqrt-softplus MoE routing with hash layers"; linear layers
//    end in Ops.SiLUMulClamp; the weighted-sum epilogue is moe_scatter_add.
//  * "Model Card for DeepSeek-V4-Flash-DSpark-FST", sections "Speeds, Sizes, Times" and
//    "Model Architecture and Objective": top-k = 6, hash routing on the first layers,
//    route_scale = 1.5, swiglu_limit = 10, one shared expert per layer, hidden 4096,
//    expert intermediate 2048.
//  * Same card, "Preprocessing" and glossary; FaStar README, "Expert virtual memory";
//    TensorSharp page, "Getting a drafter": experts are MXFP4, one E8M0 scale per 32
//    FP4 values.
//  * ds4 issue "Loader spec -- mtp.* tensor map": ffn.{gate.weight, gate.bias,
//    experts.{0..255}.{w1,w2,w3}, shared_experts.{w1,w2,w3}}.
//  * pypto deployment page, "MoE and output stages": gate -> top-6 routing -> routed and
//    shared expert FFNs -> combine.
// The exact element formats (E2M1 value table, E4M3 with round-to-nearest-even and
// saturation, E8M0 = floor(log2 amax) - emax) follow the OCP Microscaling Formats (MX)
// v1.0 specification, as the layer's contract requires.
//
// Readings taken where the pages are silent:
//  * selection uses score + bias, the weights use the unbiased score, normalised over
//    the k selected experts and multiplied by route_scale; ids are reported ascending;
//  * gate clamped from above at L, up clamped to [-L, L], h = silu(gate) * up;
//  * w1 = gate, w3 = up, w2 = down; MX blocks run along the reduction dimension;
//  * an all-zero block gets scale byte 0 (exponent -127);
//  * the shared expert reads the same MXFP8 activations and enters with weight 1;
//  * the MXFP4-activation variant (act = 1) quantises x and h with the weights' own MXFP4 rule
//    (E2M1, scale floor(log2 amax) - 2) where the layer uses MXFP8; nothing else changes.
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -fPIC -shared -pthread moe_oracle.cpp -o liboracle.so
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <fstream>
#include <functional>
#include <limits>
#include <string>
#include <thread>
#include <vector>

#include <sched.h>

namespace {

// ------------------------------------------------------------------ threads
int default_threads() {
  int n = (int)std::thread::hardware_concurrency();
  cpu_set_t set;
  if (sched_getaffinity(0, sizeof(set), &set) == 0) n = CPU_COUNT(&set);
  // cgroup v2 quota: "quota period" or "max period"
  std::ifstream f("/sys/fs/cgroup/cpu.max");
  std::string q, p;
  if (f >> q >> p && q != "max") {
    double quota = std::atof(q.c_str()), period = std::atof(p.c_str());
    if (quota > 0 && period > 0) {
      int lim = (int)std::ceil(quota / period);
      if (lim >= 1 && lim < n) n = lim;
    }
  }
  return n < 1 ? 1 : n;
}

void parallel_for(int64_t n, int threads, const std::function<void(int64_t, int64_t)>& fn) {
  if (threads <= 0) threads = default_threads();
  if (n <= 0) return;
  if (threads == 1 || n == 1) { fn(0, n); return; }
  // dynamic chunks so uneven rows (expert groups) balance
  std::atomic<int64_t> next{0};
  int64_t chunk = std::max<int64_t>(1, n / (threads * 8));
  std::vector<std::thread> pool;
  for (int t = 0; t < threads; ++t)
    pool.emplace_back([&]() {
      for (;;) {
        int64_t lo = next.fetch_add(chunk);
        if (lo >= n) break;
        fn(lo, std::min(n, lo + chunk));
      }
    });
  for (auto& th : pool) th.join();
}

// ------------------------------------------------------------------ element formats
// E2M1 (OCP MX v1.0, FP4): sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double e2m1_value(int code) {
  double v = kE2M1[code & 7];
  return (code & 8) ? -v : v;
}

// E4M3 (OCP MX v1.0, FP8): sign, 4 exponent bits (bias 7), 3 mantissa bits; S.1111.111 is NaN.
double e4m3_value(int b) {
  int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  double v = (e == 0) ? std::ldexp((double)m, -9) : std::ldexp(8.0 + m, e - 10);
  return s ? -v : v;
}

// E8M0: 2^(b - 127); 0xFF is NaN.
double e8m0_value(int b) {
  if ((b & 255) == 255) return std::numeric_limits<double>::quiet_NaN();
  return std::ldexp(1.0, (b & 255) - 127);
}

double bf16_value(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// floor(log2(a)) for finite a > 0, exact (frexp gives a = m 2^e with m in [0.5, 1)).
int floor_log2(double a) {
  int e;
  std::frexp(a, &e);
  return e - 1;
}

// round half to even of a non-negative value
double rne(double n) {
  double fl = std::floor(n), diff = n - fl;
  if (diff > 0.5) return fl + 1.0;
  if (diff < 0.5) return fl;
  return (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

// Round-to-nearest-even into E4M3 with subnormals (quantum 2^-9 below 2^-6) and saturation
// to +-448 for any finite magnitude above the largest normal; the sign of zero is kept.
uint8_t e4m3_encode(double v) {
  uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  double a = std::fabs(v);
  if (std::isnan(v)) return (uint8_t)(sign | 0x7F);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a == 0.0) return sign;
  int E = std::max(floor_log2(a), -6);
  double q = std::ldexp(1.0, E - 3);
  double val = rne(a / q) * q;
  if (val == 0.0) return sign;
  if (val >= 448.0) return (uint8_t)(sign | 0x7E);
  int E2 = floor_log2(val);
  if (E2 < -6) return (uint8_t)(sign | (uint8_t)(val / std::ldexp(1.0, -9)));
  int mant = (int)(val / std::ldexp(1.0, E2) * 8.0) - 8;
  return (uint8_t)(sign | ((E2 + 7) << 3) | mant);
}

// Round-to-nearest-even into E2M1 (grid 0, .5, 1, 1.5, 2, 3, 4, 6), saturating at +-6.
uint8_t e2m1_encode(double v) {
  uint8_t sign = std::signbit(v) ? 8 : 0;
  double a = std::fabs(v);
  if (a >= 6.0) return (uint8_t)(sign | 7);
  double q = (a < 2.0) ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
  double val = rne(a / q) * q;
  if (val > 6.0) val = 6.0;
  for (int c = 0; c < 8; ++c)
    if (kE2M1[c] == val) return (uint8_t)(sign | c);
  return (uint8_t)(sign | 7);  // unreachable
}

// Shared block exponent of an MX block: floor(log2 amax) - emax_elem, clamped to the E8M0 range;
// an all-zero block gets -127.
int mx_scale_exp(double amax, int emax_elem) {
  if (!(amax > 0.0)) return -127;
  int s = floor_log2(amax) - emax_elem;
  return std::min(127, std::max(-127, s));
}

// MXFP8 (E4M3, emax 8) quantisation of n values, blocks of 32.
void mxfp8_quantize(const double* v, int64_t n, uint8_t* q, uint8_t* s) {
  for (int64_t b = 0; b < n / 32; ++b) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(v[b * 32 + i]));
    int se = mx_scale_exp(amax, 8);
    s[b] = (uint8_t)(se + 127);
    for (int i = 0; i < 32; ++i) q[b * 32 + i] = e4m3_encode(std::ldexp(v[b * 32 + i], -se));
  }
}

// MXFP4 (E2M1, emax 2) quantisation of n values, blocks of 32; packed codes, element 2i in the low
// nibble of byte i.
void mxfp4_quantize(const double* v, int64_t n, uint8_t* codes, uint8_t* s) {
  for (int64_t b = 0; b < n / 32; ++b) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(v[b * 32 + i]));
    int se = mx_scale_exp(amax, 2);
    s[b] = (uint8_t)(se + 127);
    for (int i = 0; i < 32; i += 2) {
      uint8_t lo = e2m1_encode(std::ldexp(v[b * 32 + i], -se));
      uint8_t hi = e2m1_encode(std::ldexp(v[b * 32 + i + 1], -se));
      codes[(b * 32 + i) / 2] = (uint8_t)(lo | (hi << 4));
    }
  }
}

double mxfp8_value(const uint8_t* q, const uint8_t* s, int64_t i) { return e4m3_value(q[i]) * e8m0_value(s[i / 32]); }

double mxfp4_value(const uint8_t* codes, const uint8_t* s, int64_t i) {
  uint8_t b = codes[i / 2];
  int c = (i & 1) ? (b >> 4) : (b & 15);
  return e2m1_value(c) * e8m0_value(s[i / 32]);
}

double softplus(double l) { return std::max(l, 0.0) + std::log1p(std::exp(-std::fabs(l))); }
double silu(double z) { return z / (1.0 + std::exp(-z)); }

struct Expert {
  const uint8_t *w13, *s13, *w2, *s2;  // one expert's slices
};

Expert expert_at(const uint8_t* w13, const uint8_t* s13, const uint8_t* w2, const uint8_t* s2, int64_t e, int64_t d,
                 int64_t f) {
  Expert x;
  x.w13 = w13 + e * 2 * f * (d / 2);
  x.s13 = s13 + e * 2 * f * (d / 32);
  x.w2 = w2 + e * d * (f / 2);
  x.s2 = s2 + e * d * (f / 32);
  return x;
}

// Activation formats: the layer's MXFP8 (E4M3 codes, one byte per element) and the MXFP4 variant
// (E2M1 codes, two per byte), both with one E8M0 scale per 32 elements along the reduction dimension.
constexpr int kActMxfp8 = 0, kActMxfp4 = 1;

int64_t act_row_bytes(int act, int64_t n) { return act == kActMxfp4 ? n / 2 : n; }

double act_value(int act, const uint8_t* q, const uint8_t* s, int64_t i) {
  return act == kActMxfp4 ? mxfp4_value(q, s, i) : mxfp8_value(q, s, i);
}

// One expert applied to one activation row: gate/up dot products over d, clamp, SiLU * up,
// requantisation of h along f in the activation format, down projection over f.  hq/hs/hpre may be
// null.
void expert_row(const uint8_t* aq, const uint8_t* as, int64_t d, int64_t f, const Expert& ex, double limit, double* y,
                uint8_t* hq_out, uint8_t* hs_out, double* hpre_out, int act) {
  std::vector<double> xd(d), h(f), hd(f);
  std::vector<uint8_t> hq(act_row_bytes(act, f)), hs(f / 32);
  for (int64_t i = 0; i < d; ++i) xd[i] = act_value(act, aq, as, i);
  for (int64_t o = 0; o < f; ++o) {
    const uint8_t* wg = ex.w13 + o * (d / 2);
    const uint8_t* sg = ex.s13 + o * (d / 32);
    const uint8_t* wu = ex.w13 + (f + o) * (d / 2);
    const uint8_t* su = ex.s13 + (f + o) * (d / 32);
    double g = 0.0, u = 0.0;
    for (int64_t i = 0; i < d; ++i) {
      g += xd[i] * mxfp4_value(wg, sg, i);
      u += xd[i] * mxfp4_value(wu, su, i);
    }
    double gc = std::min(g, limit);
    double uc = std::min(std::max(u, -limit), limit);
    h[o] = silu(gc) * uc;
  }
  if (act == kActMxfp4)
    mxfp4_quantize(h.data(), f, hq.data(), hs.data());
  else
    mxfp8_quantize(h.data(), f, hq.data(), hs.data());
  for (int64_t j = 0; j < f; ++j) hd[j] = act_value(act, hq.data(), hs.data(), j);
  for (int64_t o = 0; o < d; ++o) {
    const uint8_t* wd = ex.w2 + o * (f / 2);
    const uint8_t* sd = ex.s2 + o * (f / 32);
    double acc = 0.0;
    for (int64_t j = 0; j < f; ++j) acc += hd[j] * mxfp4_value(wd, sd, j);
    y[o] = acc;
  }
  if (hq_out) std::memcpy(hq_out, hq.data(), hq.size());
  if (hs_out) std::memcpy(hs_out, hs.data(), (size_t)(f / 32));
  if (hpre_out) std::memcpy(hpre_out, h.data(), sizeof(double) * (size_t)f);
}

// Top-k of sel (descending, ties to the lower index) by repeated arg-max, or by a full sort.
void topk_indices(const std::vector<double>& sel, int64_t k, int method, std::vector<int32_t>& idx) {
  int64_t E = (int64_t)sel.size();
  idx.clear();
  if (method == 1) {
    std::vector<int32_t> order(E);
    for (int64_t e = 0; e < E; ++e) order[e] = (int32_t)e;
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return sel[a] > sel[b]; });
    idx.assign(order.begin(), order.begin() + k);
    return;
  }
  std::vector<char> taken(E, 0);
  for (int64_t j = 0; j < k; ++j) {
    int64_t best = -1;
    for (int64_t e = 0; e < E; ++e)
      if (!taken[e] && (best < 0 || sel[e] > sel[best])) best = e;
    taken[best] = 1;
    idx.push_back((int32_t)best);
  }
}

}  // namespace

extern "C" {

int orc_default_threads() { return default_threads(); }
double orc_e2m1_value(int code) { return e2m1_value(code); }
double orc_e4m3_value(int b) { return e4m3_value(b); }
double orc_e8m0_value(int b) { return e8m0_value(b); }
double orc_bf16_value(uint16_t h) { return bf16_value(h); }
int orc_mx_scale_exp(double amax, int emax_elem) { return mx_scale_exp(amax, emax_elem); }
uint8_t orc_e4m3_encode(double v) { return e4m3_encode(v); }
uint8_t orc_e2m1_encode(double v) { return e2m1_encode(v); }

void orc_e4m3_encode_many(const double* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode(v[i]);
}

// MXFP8 quantisation of rows of fp64 values (n multiple of 32).
void orc_mxfp8_quantize(const double* v, int64_t n, uint8_t* q, uint8_t* s) { mxfp8_quantize(v, n, q, s); }

// MXFP4 quantisation (E2M1, emax 2), packed codes (element 2i in the low nibble of byte i).
void orc_mxfp4_quantize(const double* v, int64_t n, uint8_t* codes, uint8_t* s) { mxfp4_quantize(v, n, codes, s); }

void orc_mxfp4_dequantize(const uint8_t* codes, const uint8_t* s, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = mxfp4_value(codes, s, i);
}

void orc_mxfp8_dequantize(const uint8_t* q, const uint8_t* s, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = mxfp8_value(q, s, i);
}

// x (bf16 [T, d]) -> activation codes [T, d] (MXFP8) or [T, d/2] (MXFP4) and scale bytes [T, d/32].
void orc_quantize_x(const uint16_t* x, int64_t T, int64_t d, uint8_t* q, uint8_t* s, int threads, int act) {
  parallel_for(T, threads, [&](int64_t lo, int64_t hi) {
    std::vector<double> row(d);
    for (int64_t t = lo; t < hi; ++t) {
      for (int64_t i = 0; i < d; ++i) row[i] = bf16_value(x[t * d + i]);
      if (act == kActMxfp4)
        mxfp4_quantize(row.data(), d, q + t * (d / 2), s + t * (d / 32));
      else
        mxfp8_quantize(row.data(), d, q + t * d, s + t * (d / 32));
    }
  });
}

// Router: logits in fp64, s = sqrt(softplus(l)), top-k on s + bias, weights = scale * s_j / sum s.
// ids ascending per token.  margin[t] = k-th largest sel minus (k+1)-th largest (inf if E == k).
// logits_out / scores_out ([T, E]) may be null.  method: 0 = repeated arg-max, 1 = full sort.
void orc_route(const uint16_t* x, int64_t T, int64_t d, const float* w, const float* bias, int64_t E, int64_t k,
               double route_scale, int method, int32_t* ids, double* wts, double* margin, double* logits_out,
               double* scores_out, int threads) {
  parallel_for(T, threads, [&](int64_t lo, int64_t hi) {
    std::vector<double> xd(d), s(E), sel(E);
    std::vector<int32_t> idx;
    for (int64_t t = lo; t < hi; ++t) {
      for (int64_t i = 0; i < d; ++i) xd[i] = bf16_value(x[t * d + i]);
      for (int64_t e = 0; e < E; ++e) {
        double l = 0.0;
        for (int64_t i = 0; i < d; ++i) l += xd[i] * (double)w[e * d + i];
        if (logits_out) logits_out[t * E + e] = l;
        s[e] = std::sqrt(softplus(l));
        sel[e] = s[e] + (double)bias[e];
        if (scores_out) scores_out[t * E + e] = s[e];
      }
      topk_indices(sel, k, method, idx);
      if (margin) {
        double kth = sel[idx[k - 1]], next = -std::numeric_limits<double>::infinity();
        std::vector<char> chosen(E, 0);
        for (int64_t j = 0; j < k; ++j) chosen[idx[j]] = 1;
        for (int64_t e = 0; e < E; ++e)
          if (!chosen[e]) next = std::max(next, sel[e]);
        margin[t] = (E == k) ? std::numeric_limits<double>::infinity() : kth - next;
      }
      std::sort(idx.begin(), idx.end());
      double sum = 0.0;
      for (int64_t j = 0; j < k; ++j) sum += s[idx[j]];
      for (int64_t j = 0; j < k; ++j) {
        ids[t * k + j] = idx[j];
        wts[t * k + j] = route_scale * s[idx[j]] / sum;
      }
    }
  });
}

// Hash router: ids = the token's table row (ascending), weights route_scale / k.
// Returns the number of tokens whose id is outside [0, V) (those rows are left untouched).
int64_t orc_hash_route(const int32_t* tok, int64_t T, const int32_t* table, int64_t V, int64_t k, double route_scale,
                       int32_t* ids, double* wts) {
  int64_t bad = 0;
  for (int64_t t = 0; t < T; ++t) {
    if (tok[t] < 0 || tok[t] >= V) { ++bad; continue; }
    std::vector<int32_t> row(table + (int64_t)tok[t] * k, table + (int64_t)tok[t] * k + k);
    std::sort(row.begin(), row.end());
    for (int64_t j = 0; j < k; ++j) {
      ids[t * k + j] = row[j];
      wts[t * k + j] = route_scale / (double)k;
    }
  }
  return bad;
}

// Token -> expert permutation: counts per expert, exclusive offsets [E+1], rows expert-major with
// tokens ascending inside an expert; perm_tok[r] = token of row r; inv_pos[t, j] = row of (t, ids[t, j]).
void orc_permute(const int32_t* ids, int64_t T, int64_t k, int64_t E, int32_t* counts, int32_t* offsets,
                 int32_t* perm_tok, int32_t* inv_pos) {
  for (int64_t e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t i = 0; i < T * k; ++i) counts[ids[i]] += 1;
  offsets[0] = 0;
  for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  for (int64_t e = 0; e < E; ++e) {
    int32_t r = offsets[e];
    for (int64_t t = 0; t < T; ++t)
      for (int64_t j = 0; j < k; ++j)
        if (ids[t * k + j] == e) {
          perm_tok[r] = (int32_t)t;
          inv_pos[t * k + j] = r;
          ++r;
        }
  }
}

// One expert on one activation row (for stage-level checks).
void orc_expert_row(const uint8_t* aq, const uint8_t* as, int64_t d, int64_t f, const uint8_t* w13,
                    const uint8_t* s13, const uint8_t* w2, const uint8_t* s2, double limit, double* y, uint8_t* hq,
                    uint8_t* hs, double* hpre, int act) {
  Expert ex{w13, s13, w2, s2};
  expert_row(aq, as, d, f, ex, limit, y, hq, hs, hpre, act);
}

// Grouped expert FFN over n_rows activation rows: row r belongs to group g where offsets[g] <= r <
// offsets[g+1] (offsets may be null: one group); y[r] = row_w[r] * expert_g(a[r]) (row_w null = 1).
// hq/hs/hpre (h codes, scales, and h before quantisation [n_rows, f]) may be null.
void orc_expert_ffn(int64_t n_rows, int64_t n_groups, const int32_t* offsets, const uint8_t* aq, const uint8_t* as,
                    int64_t d, int64_t f, const uint8_t* w13, const uint8_t* s13, const uint8_t* w2, const uint8_t* s2,
                    double limit, const double* row_w, double* y, uint8_t* hq, uint8_t* hs, double* hpre, int threads,
                    int act) {
  parallel_for(n_rows, threads, [&](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) {
      int64_t g = 0;
      if (offsets) {
        while (g < n_groups && !(offsets[g] <= r && r < offsets[g + 1])) ++g;
        if (g == n_groups) continue;
      }
      Expert ex = expert_at(w13, s13, w2, s2, g, d, f);
      expert_row(aq + r * act_row_bytes(act, d), as + r * (d / 32), d, f, ex, limit, y + r * d,
                 hq ? hq + r * act_row_bytes(act, f) : nullptr, hs ? hs + r * (f / 32) : nullptr,
                 hpre ? hpre + r * f : nullptr, act);
      double wr = row_w ? row_w[r] : 1.0;
      for (int64_t o = 0; o < d; ++o) y[r * d + o] *= wr;
    }
  });
}

// Whole layer for the tokens listed in `tokens` (n_sel of them; null = all T).  The routing is
// given (ids/wts from orc_route or orc_hash_route).  mode 0: dense per token (each (t, j) pair
// evaluated directly); mode 1: through the permutation (rows in expert-major order, then a combine).
// y_out is [n_sel, d] in the order of `tokens`.  Shared expert pointers may be null.
// The layer, optionally also returning what each (selected token, slot) row computed on the way: the h
// codes, scales and h before quantisation, [n_sel][k + 1][...] with slot k the shared expert (left
// untouched without one).  hq / hs / hpre may be null.
void orc_layer_h(const uint16_t* x, int64_t T, int64_t d, int64_t f, int64_t E, int64_t k, const int32_t* ids,
                 const double* wts, const uint8_t* w13, const uint8_t* s13, const uint8_t* w2, const uint8_t* s2,
                 const uint8_t* sh_w13, const uint8_t* sh_s13, const uint8_t* sh_w2, const uint8_t* sh_s2,
                 double limit, const int32_t* tokens, int64_t n_sel, int mode, double* y_out, int threads, int act,
                 uint8_t* hq_out, uint8_t* hs_out, double* hpre_out) {
  const int64_t hb = act_row_bytes(act, f);
  // slot (i, j) of the optional h outputs
  auto hq_at = [&](int64_t i, int64_t j) { return hq_out ? hq_out + (i * (k + 1) + j) * hb : nullptr; };
  auto hs_at = [&](int64_t i, int64_t j) { return hs_out ? hs_out + (i * (k + 1) + j) * (f / 32) : nullptr; };
  auto hp_at = [&](int64_t i, int64_t j) { return hpre_out ? hpre_out + (i * (k + 1) + j) * f : nullptr; };
  if (!tokens) n_sel = T;
  auto tok_of = [&](int64_t i) -> int64_t { return tokens ? tokens[i] : i; };
  // activations of the selected tokens (MXFP8, or MXFP4 for the FP4 variant)
  const int64_t ab = act_row_bytes(act, d);
  std::vector<uint8_t> q((size_t)n_sel * ab), s((size_t)n_sel * (d / 32));
  parallel_for(n_sel, threads, [&](int64_t lo, int64_t hi) {
    std::vector<double> row(d);
    for (int64_t i = lo; i < hi; ++i) {
      int64_t t = tok_of(i);
      for (int64_t c = 0; c < d; ++c) row[c] = bf16_value(x[t * d + c]);
      if (act == kActMxfp4)
        mxfp4_quantize(row.data(), d, &q[i * ab], &s[i * (d / 32)]);
      else
        mxfp8_quantize(row.data(), d, &q[i * ab], &s[i * (d / 32)]);
    }
  });
  std::vector<double> ysh((size_t)n_sel * d, 0.0);
  if (sh_w13) {
    Expert sh{sh_w13, sh_s13, sh_w2, sh_s2};
    parallel_for(n_sel, threads, [&](int64_t lo, int64_t hi) {
      for (int64_t i = lo; i < hi; ++i)
        expert_row(&q[i * ab], &s[i * (d / 32)], d, f, sh, limit, &ysh[i * d], hq_at(i, k), hs_at(i, k), hp_at(i, k),
                   act);
    });
  }
  if (mode == 0) {
    parallel_for(n_sel, threads, [&](int64_t lo, int64_t hi) {
      std::vector<double> ye(d);
      for (int64_t i = lo; i < hi; ++i) {
        int64_t t = tok_of(i);
        double* y = y_out + i * d;
        for (int64_t o = 0; o < d; ++o) y[o] = 0.0;
        for (int64_t j = 0; j < k; ++j) {
          Expert ex = expert_at(w13, s13, w2, s2, ids[t * k + j], d, f);
          expert_row(&q[i * ab], &s[i * (d / 32)], d, f, ex, limit, ye.data(), hq_at(i, j), hs_at(i, j), hp_at(i, j),
                     act);
          for (int64_t o = 0; o < d; ++o) y[o] += wts[t * k + j] * ye[o];
        }
        for (int64_t o = 0; o < d; ++o) y[o] += ysh[i * d + o];
      }
    });
    return;
  }
  // mode 1: build the permutation over the selected tokens, evaluate rows, combine
  std::vector<int32_t> sel_ids((size_t)n_sel * k);
  for (int64_t i = 0; i < n_sel; ++i)
    for (int64_t j = 0; j < k; ++j) sel_ids[i * k + j] = ids[tok_of(i) * k + j];
  std::vector<int32_t> counts(E), offsets(E + 1), perm((size_t)n_sel * k), inv((size_t)n_sel * k);
  orc_permute(sel_ids.data(), n_sel, k, E, counts.data(), offsets.data(), perm.data(), inv.data());
  int64_t R = n_sel * k;
  std::vector<double> yr((size_t)R * d);
  std::vector<int32_t> slot_of((size_t)R);  // routing slot j of row r (inv[i * k + j] = r)
  for (int64_t i = 0; i < n_sel; ++i)
    for (int64_t j = 0; j < k; ++j) slot_of[inv[i * k + j]] = (int32_t)j;
  parallel_for(R, threads, [&](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) {
      int64_t e = 0;
      while (!(offsets[e] <= r && r < offsets[e + 1])) ++e;
      Expert ex = expert_at(w13, s13, w2, s2, e, d, f);
      int64_t i = perm[r];
      const int64_t j = slot_of[r];
      expert_row(&q[i * ab], &s[i * (d / 32)], d, f, ex, limit, &yr[r * d], hq_at(i, j), hs_at(i, j), hp_at(i, j),
                 act);
    }
  });
  for (int64_t i = 0; i < n_sel; ++i) {
    int64_t t = tok_of(i);
    double* y = y_out + i * d;
    for (int64_t o = 0; o < d; ++o) y[o] = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      const double* src = &yr[(int64_t)inv[i * k + j] * d];
      for (int64_t o = 0; o < d; ++o) y[o] += wts[t * k + j] * src[o];
    }
    for (int64_t o = 0; o < d; ++o) y[o] += ysh[i * d + o];
  }
}

void orc_layer(const uint16_t* x, int64_t T, int64_t d, int64_t f, int64_t E, int64_t k, const int32_t* ids,
               const double* wts, const uint8_t* w13, const uint8_t* s13, const uint8_t* w2, const uint8_t* s2,
               const uint8_t* sh_w13, const uint8_t* sh_s13, const uint8_t* sh_w2, const uint8_t* sh_s2,
               double limit, const int32_t* tokens, int64_t n_sel, int mode, double* y_out, int threads, int act) {
  orc_layer_h(x, T, d, f, E, k, ids, wts, w13, s13, w2, s2, sh_w13, sh_s13, sh_w2, sh_s2, limit, tokens, n_sel, mode,
              y_out, threads, act, nullptr, nullptr, nullptr);
}

}  // extern "C"
