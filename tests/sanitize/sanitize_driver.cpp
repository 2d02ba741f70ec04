// Runs the oracle end to end on a small seeded layer, for a build instrumented with AddressSanitizer and
// UndefinedBehaviorSanitizer (tests/test_sanitizers.py compiles it with the oracle and the generator).
#include <cstdint>
#include <cstdio>
#include <vector>

extern "C" {
void synth_x_bf16(uint64_t seed, int64_t T, int64_t d, double scale, const int32_t* attempt, uint16_t* out, int threads);
void synth_router(uint64_t seed, int64_t E, int64_t d, float* w, float* b);
void synth_mxfp4(uint64_t seed, int sc, int ss, int64_t row0, int64_t rows, int64_t cols, int64_t d_in,
                 uint8_t* codes, uint8_t* scales, int threads);
void synth_token_ids(uint64_t seed, int64_t T, int64_t V, int32_t* tok);
void synth_hash_table(uint64_t seed, int64_t V, int64_t E, int64_t k, int32_t* table);
void orc_route(const uint16_t* x, int64_t T, int64_t d, const float* w, const float* bias, int64_t E, int64_t k,
               double route_scale, int method, int32_t* ids, double* wts, double* margin, double* logits_out,
               double* scores_out, int threads);
int64_t orc_hash_route(const int32_t* tok, int64_t T, const int32_t* table, int64_t V, int64_t k, double route_scale,
                       int32_t* ids, double* wts);
void orc_permute(const int32_t* ids, int64_t T, int64_t k, int64_t E, int32_t* counts, int32_t* offsets,
                 int32_t* perm_tok, int32_t* inv_pos);
void orc_layer(const uint16_t* x, int64_t T, int64_t d, int64_t f, int64_t E, int64_t k, const int32_t* ids,
               const double* wts, const uint8_t* w13, const uint8_t* s13, const uint8_t* w2, const uint8_t* s2,
               const uint8_t* sh_w13, const uint8_t* sh_s13, const uint8_t* sh_w2, const uint8_t* sh_s2,
               double limit, const int32_t* tokens, int64_t n_sel, int mode, double* y_out, int threads, int act);
}

int main() {
  const int64_t T = 16, d = 256, f = 128, E = 8, k = 2, V = 100;
  const int threads = 2;
  std::vector<uint16_t> x(T * d);
  synth_x_bf16(0, T, d, 1.0, nullptr, x.data(), threads);
  std::vector<float> w(E * d), b(E);
  synth_router(0, E, d, w.data(), b.data());
  std::vector<uint8_t> w13(E * 2 * f * d / 2), s13(E * 2 * f * d / 32), w2(E * d * f / 2), s2(E * d * f / 32);
  synth_mxfp4(0, 4, 9, 0, E * 2 * f, d, d, w13.data(), s13.data(), threads);
  synth_mxfp4(0, 11, 12, 0, E * d, f, d, w2.data(), s2.data(), threads);
  std::vector<uint8_t> h13(2 * f * d / 2), hs13(2 * f * d / 32), h2(d * f / 2), hs2(d * f / 32);
  synth_mxfp4(0, 5, 10, 0, 2 * f, d, d, h13.data(), hs13.data(), threads);
  synth_mxfp4(0, 13, 14, 0, d, f, d, h2.data(), hs2.data(), threads);
  std::vector<int32_t> ids(T * k);
  std::vector<double> wts(T * k), margin(T), logits(T * E), scores(T * E);
  for (int method = 0; method < 2; ++method)
    orc_route(x.data(), T, d, w.data(), b.data(), E, k, 1.5, method, ids.data(), wts.data(), margin.data(),
              logits.data(), scores.data(), threads);
  std::vector<int32_t> counts(E), offsets(E + 1), perm(T * k), inv(T * k);
  orc_permute(ids.data(), T, k, E, counts.data(), offsets.data(), perm.data(), inv.data());
  std::vector<double> y(T * d), y2(T * d), y4(T * d), y42(T * d);
  for (int mode = 0; mode < 2; ++mode) {
    orc_layer(x.data(), T, d, f, E, k, ids.data(), wts.data(), w13.data(), s13.data(), w2.data(), s2.data(),
              h13.data(), hs13.data(), h2.data(), hs2.data(), 10.0, nullptr, 0, mode, mode ? y2.data() : y.data(),
              threads, 0);
    orc_layer(x.data(), T, d, f, E, k, ids.data(), wts.data(), w13.data(), s13.data(), w2.data(), s2.data(),
              h13.data(), hs13.data(), h2.data(), hs2.data(), 10.0, nullptr, 0, mode, mode ? y42.data() : y4.data(),
              threads, 1);
  }
  std::vector<int32_t> tok(T), table(V * k), hids(T * k);
  std::vector<double> hw(T * k);
  synth_token_ids(0, T, V, tok.data());
  synth_hash_table(0, V, E, k, table.data());
  if (orc_hash_route(tok.data(), T, table.data(), V, k, 1.5, hids.data(), hw.data()) != 0) return 2;
  for (int64_t i = 0; i < T * d; ++i)
    if (y[i] != y2[i] || y4[i] != y42[i]) return 3;  // dense and permuted evaluation agree bit for bit
  std::printf("ok\n");
  return 0;
}
