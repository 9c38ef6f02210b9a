// Host-side layout and optimizer arithmetic (see host_math.cpp).
#pragma once

#include <cstdint>
#include <vector>

#include "../../include/mt.h"

namespace mt {

constexpr int64_t kAlign = 64;  // tensor offsets are multiples of 64 elements

struct TensorDesc {
  int unit, kind;
  int64_t offset, rows, cols;
  char name[24];
};

// Offsets of a layer's tensors relative to the start of its unit.
struct LayerOffsets {
  int64_t attn_norm, wqkv, wo, mlp_norm, wgu, wdown;
};

struct FlatLayout {
  std::vector<TensorDesc> tensors;
  std::vector<int64_t> unit_off, unit_len;  // L + 2 units
  int64_t embed = 0;                        // absolute offset of the embedding
  LayerOffsets layer{};                     // per-layer relative offsets
  int64_t final_norm = 0, head = 0;         // relative to the head unit
  int64_t n_total = 0, max_unit = 0;
};

bool config_valid(const mt_config& c, const char** why);
FlatLayout build_layout(const mt_config& c);

uint16_t to_bf16_rne(float f);
void emit_bf16(const float* src, uint16_t* dst, int64_t n, int threads);

struct AdamArgs {
  float *w, *m, *v;
  float* grad_out;          // receives the gradient (may be null)
  const float* grad_in;     // fp32 gradient when slab is null
  const uint16_t* slab;     // bf16 gradient (takes precedence)
  uint16_t* store;          // bf16 copy of the updated weights (may be null)
  int64_t n, t;
  float lr, beta1, beta2, eps;
  bool apply;               // false: only write grad_out
  bool accumulate = false;  // gradient = grad_out (running sum) + this gradient
  float grad_scale = 1.f;   // Adam (and grad_out when applying) use gradient * grad_scale
};

void adam_pass(const AdamArgs& a, int threads);
int default_threads();

}  // namespace mt
