// select_mlp.cu -- the learned variant selector on the host.
//
// Method: "Leveraging Large-Scale Data for Efficient Low-Bit CUTLASS GEMM
// Optimization via Neural Networks" (press summary page), section 3: a
// feed-forward network maps (M, N, K, SM count) to one of the nine templates;
// this file loads such a network (weights trained offline by
// bit_tensor_gemm_gb300/selector_mlp.py on sweep timings from this GPU) and
// evaluates it in float32: standardised inputs (log2 M, log2 N, log2 K, SM
// count), ReLU hidden layers, argmax of the output layer.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "lbgemm.h"

namespace lbg {
lbgemm_status report_error(lbgemm_status st, const char* message);

namespace {

struct Layer {
  int n_in = 0, n_out = 0;
  std::vector<float> W;  // n_out x n_in, row-major
  std::vector<float> b;
};

struct Mlp {
  bool loaded = false;
  float mean[4] = {0, 0, 0, 0};
  float stdv[4] = {1, 1, 1, 1};
  std::vector<Layer> layers;
};

std::mutex g_mu;
Mlp g_models[9];  // indexed by bits (1, 4, 8)

bool parse(FILE* f, Mlp& m, int& bits, std::string& why) {
  char word[64];
  int version = 0;
  if (fscanf(f, "%63s %d", word, &version) != 2 || strcmp(word, "lbgemm-mlp") != 0 ||
      version != 1) {
    why = "not an lbgemm-mlp version 1 file";
    return false;
  }
  if (fscanf(f, "%63s %d", word, &bits) != 2 || strcmp(word, "bits") != 0 ||
      (bits != 1 && bits != 4 && bits != 8)) {
    why = "bad bits line";
    return false;
  }
  if (fscanf(f, "%63s", word) != 1 || strcmp(word, "norm") != 0) {
    why = "missing norm line";
    return false;
  }
  for (int i = 0; i < 4; ++i)
    if (fscanf(f, "%f", &m.mean[i]) != 1) {
      why = "bad norm means";
      return false;
    }
  for (int i = 0; i < 4; ++i)
    if (fscanf(f, "%f", &m.stdv[i]) != 1 || !(m.stdv[i] > 0.0f)) {
      why = "bad norm deviations";
      return false;
    }
  int L = 0;
  if (fscanf(f, "%63s %d", word, &L) != 2 || strcmp(word, "layers") != 0 || L < 1 || L > 16) {
    why = "bad layers line";
    return false;
  }
  int prev = 4;
  for (int l = 0; l < L; ++l) {
    Layer ly;
    if (fscanf(f, "%63s %d %d", word, &ly.n_in, &ly.n_out) != 3 || strcmp(word, "layer") != 0 ||
        ly.n_in != prev || ly.n_out < 1 || ly.n_out > 4096) {
      why = "bad layer header";
      return false;
    }
    ly.W.resize((size_t)ly.n_in * ly.n_out);
    ly.b.resize(ly.n_out);
    for (auto& w : ly.W)
      if (fscanf(f, "%f", &w) != 1) {
        why = "truncated weights";
        return false;
      }
    for (auto& v : ly.b)
      if (fscanf(f, "%f", &v) != 1) {
        why = "truncated biases";
        return false;
      }
    prev = ly.n_out;
    m.layers.push_back(std::move(ly));
  }
  m.loaded = true;
  return true;
}

// Top two classes of the network for one input (second = -1 with one class).
void forward(const Mlp& m, const float x_in[4], int& first, int& second) {
  std::vector<float> h(4), nxt;
  for (int i = 0; i < 4; ++i) h[i] = (x_in[i] - m.mean[i]) / m.stdv[i];
  for (size_t l = 0; l < m.layers.size(); ++l) {
    const Layer& ly = m.layers[l];
    nxt.assign(ly.n_out, 0.0f);
    for (int o = 0; o < ly.n_out; ++o) {
      float s = ly.b[o];
      for (int i = 0; i < ly.n_in; ++i) s += ly.W[(size_t)o * ly.n_in + i] * h[i];
      nxt[o] = (l + 1 < m.layers.size() && s < 0.0f) ? 0.0f : s;
    }
    h.swap(nxt);
  }
  first = 0;
  for (int o = 1; o < (int)h.size(); ++o)
    if (h[o] > h[first]) first = o;
  second = -1;
  for (int o = 0; o < (int)h.size(); ++o)
    if (o != first && (second < 0 || h[o] > h[second])) second = o;
}

}  // namespace

// Variant the loaded network picks for a shape, or -1 when no nine-class
// network is loaded for `bits`.
int mlp_pick(int bits, int64_t M, int64_t N, int64_t K, int sm_count) {
  if (bits < 0 || bits > 8) return -1;
  std::lock_guard<std::mutex> lock(g_mu);
  const Mlp& m = g_models[bits];
  if (!m.loaded || m.layers.back().n_out != 9) return -1;
  // a network trained on one SM count (its SM feature constant: standard
  // deviation stored as 1) answers for that SM count only
  if (m.stdv[3] == 1.0f && std::fabs((float)sm_count - m.mean[3]) > 0.5f) return -1;
  const float x[4] = {(float)std::log2((double)M), (float)std::log2((double)N),
                      (float)std::log2((double)K), (float)sm_count};
  int a, b;
  forward(m, x, a, b);
  return a;
}

// Loads a network file (no default loading first: the defaults use this).
lbgemm_status mlp_load_file(const char* path) {
  if (!path) return report_error(LBGEMM_ERR_INVALID_ARG, "null path");
  FILE* f = fopen(path, "r");
  if (!f) return report_error(LBGEMM_ERR_INVALID_ARG, "cannot open the network file");
  Mlp m;
  int bits = 0;
  std::string why;
  const bool ok = parse(f, m, bits, why);
  fclose(f);
  if (!ok) return report_error(LBGEMM_ERR_INVALID_ARG, ("network file: " + why).c_str());
  std::lock_guard<std::mutex> lock(g_mu);
  g_models[bits] = std::move(m);
  return LBGEMM_OK;
}

// The shipped table and networks are loaded before any change the caller
// makes (api.cu).
void ensure_defaults();

}  // namespace lbg

extern "C" {

lbgemm_status lbgemm_mlp_load(const char* path) {
  lbg::ensure_defaults();
  return lbg::mlp_load_file(path);
}

lbgemm_status lbgemm_mlp_clear(void) {
  lbg::ensure_defaults();
  std::lock_guard<std::mutex> lock(lbg::g_mu);
  for (auto& m : lbg::g_models) m = lbg::Mlp();
  return LBGEMM_OK;
}

int lbgemm_mlp_predict(int bits, int64_t M, int64_t N, int64_t K, int sm_count, int* second) {
  if ((bits != 1 && bits != 4 && bits != 8) || M < 1 || N < 1 || K < 1) return -1;
  lbg::ensure_defaults();
  std::lock_guard<std::mutex> lock(lbg::g_mu);
  const lbg::Mlp& m = lbg::g_models[bits];
  if (!m.loaded) return -1;
  const float x[4] = {(float)std::log2((double)M), (float)std::log2((double)N),
                      (float)std::log2((double)K), (float)sm_count};
  int a, b;
  lbg::forward(m, x, a, b);
  if (second) *second = b;
  return a;
}

}  // extern "C"
